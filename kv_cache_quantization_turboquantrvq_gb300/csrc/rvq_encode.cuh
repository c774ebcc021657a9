// rvq_encode.cuh - TurboQuantRVQ encode+pack device code for sm_103a, shared
// by the encode kernels (rvq.cu) and the fused decode-time flush (flush.cu).
// Each body runs one CTA's share of a persistent grid: CTA `cta` of `ncta`.
//
// Method (VeloxQuant-MLX blog, tag "rvq", "The pipeline, as it actually runs"
// and "What 'quantize' means here, precisely"; rotation as in tag
// "turboquant", "Kernel 3: Fused Hadamard + Quantize"), per key row x of
// D = 128 fp16 values:
//   n = ||x||, y = H (x / n) / sqrt(D)           normalise + Walsh-Hadamard
//   i1 = #{k : y > b1_k},  r = y - c1[i1]          stage 1 + residual
//   i2 = #{k : r > b2_k}                           stage 2
//   packed1/packed2: LSB-first b-bit codes in uint32 words, plus the norm.
// The pages fuse quantize->pack after a separate rotation dispatch; here the
// norm, rotation, both stages and both packs are one pass over HBM.
//
// Encode design (two threads per row, 16-row blocks per warp, 16 warps/SM):
//  * each warp owns a private 2-stage ring of 16-row blocks in shared memory,
//    each block two TMA tensor boxes (16 rows x 64 channels, one per input
//    half) that complete on an mbarrier and land with the 128-byte swizzle
//    (chunk c of row r at chunk c ^ (r & 7)), so 16-byte row reads are free of
//    bank conflicts;
//  * lane l takes row l & 15 and input half h = l >> 4: with
//    H = [[H64, H64], [H64, -H64]] it computes Z_h = H64 x_h on its own 64
//    values (the first butterfly fused with the fp16 -> fp32 conversion,
//    then five fp32x2 stages), swaps Z_h with its partner (lane l ^ 16) by
//    shuffles and keeps Z_0 + Z_1 or Z_0 - Z_1: its 64 output coordinates;
//    the norm comes from the partners' sums of squares (Parseval);
//  * the quantizer is unrolled over those 64 coordinates, in registers: the
//    symmetric 1/2-bit codebooks take sign-bit arithmetic (no tables), other
//    codebooks the shuffle-table count (GridTable in launch.h) or a plain
//    count; each thread stores its half of the row's words (the 16 rows x 2
//    halves of a block are contiguous in global memory);
//  * every code is kept unless its pre-quantization value lies within a guard
//    band of a boundary; such rows are redone by the whole warp in exact /
//    double-float arithmetic (rvq_fixup_row), so the packed words equal those
//    of exact arithmetic.
// The library's books (symmetric 4-level books, b = 2, and 16-level books
// with a pair table, b = 4) have an encoder of their own with the rotation on
// the 5th-generation tensor cores: rvq_encode_tm_body, further below.
//
// The including translation unit defines VQ_RVQ_ERR, the device error word
// the bodies report into (VQ_DEVERR_* bits).
#pragma once

#include <cuda_fp16.h>

#include "device_common.cuh"
#include "launch.h"
#include "tcgen05.cuh"

#ifndef VQ_RVQ_ERR
#error "define VQ_RVQ_ERR (the device error word) before including rvq_encode.cuh"
#endif

namespace vq {
namespace {


// the key/value row (shared with the other codec's device code when both
// are included in one translation unit)
#ifndef VQ_ROW_CONSTANTS_DEFINED
#define VQ_ROW_CONSTANTS_DEFINED
constexpr int D = 128;
constexpr int ROW_BYTES = D * 2;
constexpr int ROW_STRIDE = ROW_BYTES + 16;
#endif

// Encoder shared memory: the input rings of all warps (1024-byte aligned
// 4 KB blocks of ER = 16 rows), then, for the table-driven quantizers only,
// per warp a slice scratch (enc_pairs coordinate pairs x 32 lanes) and a
// per-lane word staging row (stride WL + 1 words per stream).  The symmetric
// 1/2-bit quantizer is unrolled over a thread's 64 coordinates in registers
// (small enough for the instruction cache); the 16-level table quantizer is
// not, so it runs a rolled loop over slices of the half row.
constexpr int ER = 16;
constexpr int ENC_STAGES = 2;
constexpr int ENC_BLOCK = ER * ROW_BYTES;  // two swizzled 2 KB boxes
constexpr int SMEM_MAX = 227 * 1024;
enum { MODE_PLAIN = 0, MODE_GRID = 1, MODE_SYM = 2, MODE_PAIR = 3 };
__host__ __device__ constexpr int enc_pairs(int bits) { return 32 / bits > 8 ? 32 / bits : 8; }
__host__ __device__ constexpr int enc_warp_bytes(int bits, int mode)
{
    return ENC_STAGES * (ENC_BLOCK + 8) +
           (mode == MODE_SYM ? 0 : enc_pairs(bits) * 32 * 8 + 2 * 32 * (D * bits / 64 + 1) * 4);
}
// The table-driven quantizer reads its cell tables from shared memory,
// replicated per lane (entry g of lane l at g * 32 + l: conflict-free): stage 1
// {boundary, code below it, centroid below, centroid step} (16 bytes), stage 2
// {boundary, code below it} (8 bytes).
constexpr int ENC_TAB_BYTES = 32 * 32 * 16 + 32 * 32 * 8;
__host__ __device__ constexpr int enc_tab_bytes(int mode)
{
    return mode == MODE_GRID ? ENC_TAB_BYTES : 0;
}
// sign masks of the randomised rotation (2 halves x 8 chunks x 16 B), padded so
// that the TMA rings after them stay 1024-byte aligned (128-byte swizzle)
constexpr int ENC_SGN_BYTES = 1024;
__host__ __device__ constexpr int enc_warps(int bits, int mode)
{
    return (SMEM_MAX - 1024 - enc_tab_bytes(mode) - ENC_SGN_BYTES) / enc_warp_bytes(bits, mode) > 16
               ? 16
               : (SMEM_MAX - 1024 - enc_tab_bytes(mode) - ENC_SGN_BYTES) / enc_warp_bytes(bits, mode);
}
__host__ __device__ constexpr int enc_smem(int bits, int mode)
{
    return 1024 + enc_tab_bytes(mode) + ENC_SGN_BYTES + enc_warps(bits, mode) * enc_warp_bytes(bits, mode);
}

// sqrt(128) = 8 sqrt(2) as a double-float (nearest fp32 + fp32 remainder).
constexpr float SQRT_D_HI = 11.313708305358887f;
constexpr float SQRT_D_LO = 1.936258797741175e-07f;
constexpr float GRID_MAGIC = 12582912.0f;  // 1.5 * 2^23: fma(u, 31, M) puts RN(31u) in the low bits

__device__ __forceinline__ int grid_cell(float v, float a, float bc)
{
    const float u = __saturatef(fmaf(v, a, bc));
    return __float_as_int(fmaf(u, 31.0f, GRID_MAGIC));  // low 5 bits = cell; shuffles use only those
}

// Boundary count of v in one stage.  GRID: table lookup (exact count for the
// fp32 v); otherwise a plain count over the boundaries.  `m` tracks the
// distance to the nearest boundary that could be decisive.
template <int BITS, bool GRID>
__device__ __forceinline__ int stage_code(float v, float tb, int tc, const GridTable &t,
                                          const float *b, float &m)
{
    if constexpr (GRID) {
        const int g = grid_cell(v, t.a, t.bc);
        const float bnd = __shfl_sync(FULL_MASK, tb, g);
        const int cl = __shfl_sync(FULL_MASK, tc, g);
        // v > bnd exactly when bnd - v is negative (an exact tie gives +0):
        // the increment is that sign bit
        const float d = bnd - v;
        m = fminf(m, fabsf(d));
        return cl + (int)(__float_as_uint(d) >> 31);
    } else {
        // fallback for codebooks without a grid table: a plain loop over the
        // boundaries (uniform across the warp), kept rolled to bound code size
        int code = 0;
#pragma unroll 1
        for (int k = 0; k < (1 << BITS) - 1; ++k) {
            const float d = b[k] - v;
            m = fminf(m, fabsf(d));
            code += (int)(__float_as_uint(d) >> 31);
        }
        return code;
    }
}

// Exact boundary count of the double-float value (vh + vl).
template <int BITS, bool GRID>
__device__ __forceinline__ int stage_code_df(float vh, float vl, float tb, int tc,
                                             const GridTable &t, const float *b)
{
    if constexpr (GRID) {
        const int g = grid_cell(vh, t.a, t.bc);
        const float bnd = __shfl_sync(FULL_MASK, tb, g);
        const int cl = __shfl_sync(FULL_MASK, tc, g);
        return cl + ((vh > bnd || (vh == bnd && vl > 0.0f)) ? 1 : 0);
    } else {
        int code = 0;
#pragma unroll 1
        for (int k = 0; k < (1 << BITS) - 1; ++k)
            code += (vh > b[k] || (vh == b[k] && vl > 0.0f)) ? 1 : 0;
        return code;
    }
}

// Both stages of one coordinate from the shared-memory cell tables: the
// stage-1 entry carries the boundary of the cell, the code below it and the
// centroids on both sides, so the residual needs no further lookup; two
// table reads per coordinate instead of five shuffles.  v > bnd exactly when
// bnd - v is negative (an exact tie gives +0), and the centroid step is taken
// with the saturated multiple of the same difference.
__device__ __forceinline__ void grid2_code(float v, const GridTable &ta, const GridTable &tb,
                                           const unsigned char *t1l, const unsigned char *t2l, int &c1,
                                           int &c2, float &m)
{
    const float u1 = __saturatef(fmaf(v, ta.a, ta.bc));
    // cell in [0, 31]: u1 is saturated (NaN saturates to 0)
    const uint32_t g1 = __float_as_uint(fmaf(u1, 31.0f, GRID_MAGIC)) - 0x4B400000u;
    const float4 e1 = *reinterpret_cast<const float4 *>(t1l + g1 * 512u);
    const float d1 = e1.x - v;
    m = fminf(m, fabsf(d1));
    c1 = __float_as_int(e1.y) + (int)(__float_as_uint(d1) >> 31);
    const float s1 = __saturatef(d1 * -1.2676506e30f);  // 1 when v > bnd
    const float r = fmaf(-s1, e1.w, v - e1.z);
    const float u2 = __saturatef(fmaf(r, tb.a, tb.bc));
    const uint32_t g2 = __float_as_uint(fmaf(u2, 31.0f, GRID_MAGIC)) - 0x4B400000u;
    const float2 e2 = *reinterpret_cast<const float2 *>(t2l + g2 * 256u);
    const float d2 = e2.x - r;
    m = fminf(m, fabsf(d2));
    c2 = __float_as_int(e2.y) + (int)(__float_as_uint(d2) >> 31);
}

// Symmetric 1- and 2-bit codebooks (c[k] = -c[L-1-k], middle boundary 0) are
// quantized without tables: |y| is compared with the one positive boundary and
// the code bits are sign bits.  Codes are built MSB-first by left funnel
// shifts of sign bits, elements of a word in reverse order, and the word is
// complemented at the end (the sign bit is the complement of "greater").
//   b = 2:  i = y > 0 ? 2 + u : 1 - u,  u = |y| > B   (bits: !sgn(y), !(sgn(y) ^ sgn(|y| - B)))
//   b = 1:  i = y > 0                                   (bit: !sgn(y))
// The residual of stage 1 is r = sgn(y) (|y| - c) with c the positive centroid.
// Per-row constants of the symmetric quantizers, in units of S = H x (the
// unnormalised transform, S = y n sqrt(D)): the positive boundaries B and E
// of the two stages, B - c2, dc = c3 - c2 and (b = 1) c1, each scaled by
// den = n sqrt(D); for b = 2 also k1 = 2 / B and k2 = 2 / E and the margin
// thresholds G1 = g (B + 2g) and G2 = g (E + 2g), g the guard band in the
// same units.
struct SymRow {
    float bb, be, bc2, dc, c1, k1, k2, G1, G2;
};

// Two coordinates (a pair, both of one row) of the symmetric b = 2 quantizer.
// t2 = |y| - B is positive exactly when |y| > B.  The centroid step uses a
// saturated multiply (1 when t2 > 0, 0 when t2 <= 0), which keeps the
// selection on the FMA pipe; ra = |y| - c(i) and t4 = |ra| - E likewise for
// stage 2.  The codes come from two bits of z1 = y k1 and of z2 = ra k2: the
// sign, and bit 30 (the top exponent bit of an fp32 value, set exactly when
// |z| >= 2, i.e. |y| >= B or |ra| >= E).  One funnel shift by 2 moves both
// into the accumulating word (bit 2i + 1: sign, bit 2i: the "outer" bit), and
// sym2_words turns those into the codes with whole-word logic.
// Margins: a value within g of a boundary of stage 1 (0 or B) has
// |y t2| < g (B + g), and one within g of a boundary of stage 2 has
// |ra t4| < g (E + g); m1 and m2 keep the running minima of those products,
// and a row whose minimum is below G1 = g (B + 2g) or G2 (the extra g covers
// the products' rounding) takes the exact path.  Conversely a coordinate of an
// unflagged row is at least g from every boundary, which is what the bit-30
// test needs: z rounds within a few ulps of the exact ratio, so that bit can
// differ from the sign of t2 (t4) only within 2^-21 B (E) of the boundary,
// and the symmetric mode is chosen only for B, E < 1/4.  A value exactly on
// a boundary, and y = 0, give a zero product.
__device__ __forceinline__ void sym2_code2(float2 y, const SymRow &k, uint32_t &a1x, uint32_t &a2x,
                                           uint32_t &a1y, uint32_t &a2y, float &m1, float &m2)
{
    const float2 t2 = make_float2(fabsf(y.x) - k.bb, fabsf(y.y) - k.bb);
    const float2 su = make_float2(__saturatef(t2.x * 1.2676506e30f), __saturatef(t2.y * 1.2676506e30f));  // 2^100
    // |y| - c2 = (|y| - B) + (B - c2)
    const float2 ya = __fadd2_rn(t2, make_float2(k.bc2, k.bc2));
    const float2 ra = __ffma2_rn(make_float2(-k.dc, -k.dc), su, ya);
    const float2 t4 = make_float2(fabsf(ra.x) - k.be, fabsf(ra.y) - k.be);
    const float2 p1 = __fmul2_rn(y, t2);
    const float2 p2 = __fmul2_rn(ra, t4);
    m1 = fminf(fminf(m1, fabsf(p1.x)), fabsf(p1.y));
    m2 = fminf(fminf(m2, fabsf(p2.x)), fabsf(p2.y));
    const float2 z1 = __fmul2_rn(y, make_float2(k.k1, k.k1));
    const float2 z2 = __fmul2_rn(ra, make_float2(k.k2, k.k2));
    a1x = __funnelshift_l(__float_as_uint(z1.x), a1x, 2);
    a2x = __funnelshift_l(__float_as_uint(z2.x), a2x, 2);
    a1y = __funnelshift_l(__float_as_uint(z1.y), a1y, 2);
    a2y = __funnelshift_l(__float_as_uint(z2.y), a2y, 2);
}

// Code words of 16 coordinates from the accumulated (sign, outer) bit pairs
// of sym2_code2.  Stage 1: bit 1 = [y >= 0] = NOT sign(y), bit 0 = [y >= 0]
// XOR [|y| < B] = sign(y) XOR outer.  Stage 2 (residual r = sgn(y) ra): bit 1
// = NOT (sign(y) XOR sign(ra)), bit 0 = its XOR with NOT outer2; with
// v = a2 XOR (a1 AND the sign positions) both words have the form
// f(v) = (NOT v on odd bits) | ((v XOR v >> 1) on even bits).
__device__ __forceinline__ uint32_t sym2_pairs_to_codes(uint32_t v)
{
    return (~v & 0xAAAAAAAAu) | ((v ^ (v >> 1)) & 0x55555555u);
}
__device__ __forceinline__ void sym2_words(uint32_t a1, uint32_t a2, uint32_t &w1, uint32_t &w2)
{
    w1 = sym2_pairs_to_codes(a1);
    w2 = sym2_pairs_to_codes(a2 ^ (a1 & 0xAAAAAAAAu));
}

__device__ __forceinline__ void sym1_code(float y, const SymRow &k, uint32_t &a1, uint32_t &a2, float &m)
{
    const float r = y - copysignf(k.c1, y);
    m = fminf(m, fabsf(y));
    m = fminf(m, fabsf(r));
    a1 = __funnelshift_l(__float_as_uint(y), a1, 1);
    a2 = __funnelshift_l(__float_as_uint(r), a2, 1);
}

// Destination row of source row `row`; false if its batch offset is invalid.
__device__ __forceinline__ bool rvq_dst_row(const RvqEncodeParams &p, int row, size_t &drow)
{
    const int bh = fdiv(p.divS, row);
    const int s = row - bh * p.S;
    if (s >= p.S_q) return false;  // a token of the fp16 window (fused flush)
    int off = 0;
    if (p.dst_off != nullptr) {
        off = __ldg(p.dst_off + fdiv(p.divH, bh));
        if (off < 0 || off > p.S_dst - p.S_q) {
            atomicOr(&VQ_RVQ_ERR, (unsigned)VQ_DEVERR_BAD_OFFSET);
            return false;
        }
    }
    drow = (size_t)bh * p.S_dst + off + s;
    return true;
}

__device__ __forceinline__ void wht_lane_exact(float (&a)[4], int lane)
{
    // bits 0-1 of the coordinate index live in the register index
    float t0 = a[0] + a[1], t1 = a[0] - a[1], t2 = a[2] + a[3], t3 = a[2] - a[3];
    a[0] = t0 + t2; a[1] = t1 + t3; a[2] = t0 - t2; a[3] = t1 - t3;
    // bits 2-6 live in the lane index
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
        const bool upper = (lane & m) != 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float o = __shfl_xor_sync(FULL_MASK, a[j], m);
            a[j] = upper ? (o - a[j]) : (a[j] + o);
        }
    }
}

// Whole-warp recompute of one row in exact / double-float arithmetic.
// Lane l handles coordinates 4l..4l+3.
//  * S = H x exactly: x is split into three pieces on power-of-two grids
//    (q1 = 2^(e-15), q2 = 2^(e-32), the rest, e = exponent of max|x|) whose
//    Hadamard sums all fit in 24 bits, so each piece's transform is exact in
//    fp32 and S = S1 + S2 + S3 exactly.
//  * Q = sum x^2 in double-float (squares of fp16 values are exact in fp32),
//    n = sqrt(Q) and 1/(n sqrt(D)) in double-float.
//  * y = S / (n sqrt(D)) in double-float (about 2^-44 relative), and each
//    boundary count is taken on the double-float value.
// The row's raw values are read from the staged block (row r of it, global
// row `row`); its words and norm go straight to global memory.
// HALF: bytes between the staged block's two 64-coordinate halves (16-row
// blocks: ENC_BLOCK / 2); HALF = 0: the row is read from global memory (the
// input, p.x), where it is contiguous.
template <int BITS, bool GRID, int HALF = ENC_BLOCK / 2>
__device__ __noinline__ void rvq_fixup_row(const RvqEncodeParams &p, const unsigned char *sblk,
                                           int r, int row, int lane, float tb1, int tc1, float tb2,
                                           int tc2, float tcen)
{
    constexpr int E = 32 / BITS;
    constexpr int W = D * BITS / 32;
    constexpr int LPW = E / 4;  // lanes per packed word
    // x[4l .. 4l+3]: box l >> 4, 16-byte chunk (l & 15) >> 1, half (l & 1)
    uint2 raw;
    if constexpr (HALF == 0)
        raw = __ldg(reinterpret_cast<const uint2 *>(static_cast<const unsigned char *>(p.x) + (size_t)row * ROW_BYTES) + lane);
    else
        raw = *reinterpret_cast<const uint2 *>(sblk + (lane >> 4) * HALF + swz128(r, (lane & 15) >> 1) + 8 * (lane & 1));
    if (p.has_sgn) {
        raw.x ^= half2_sign_mask(sign_pair(p.sgn, 4 * lane));
        raw.y ^= half2_sign_mask(sign_pair(p.sgn, 4 * lane + 2));
    }
    const __half2 h01 = *reinterpret_cast<const __half2 *>(&raw.x);
    const __half2 h23 = *reinterpret_cast<const __half2 *>(&raw.y);
    float x[4] = {__low2float(h01), __high2float(h01), __low2float(h23), __high2float(h23)};

    // row max |x| and sum of squares (double-float)
    float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
    float qh = x[0] * x[0], ql = 0.0f;
#pragma unroll
    for (int j = 1; j < 4; ++j) {
        float s, e;
        two_sum(qh, x[j] * x[j], s, e);
        qh = s;
        ql += e;
    }
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) {
        amax = fmaxf(amax, __shfl_xor_sync(FULL_MASK, amax, m));
        const float oh = __shfl_xor_sync(FULL_MASK, qh, m);
        const float ol = __shfl_xor_sync(FULL_MASK, ql, m);
        float s, e;
        two_sum(qh, oh, s, e);
        e += ql + ol;
        fast_two_sum(s, e, qh, ql);
    }

    // n = sqrt(Q), den = n sqrt(D), inv = 1/den, all double-float
    float nh = 0.0f, nl = 0.0f, ih = 0.0f, il = 0.0f;
    if (qh > 0.0f) {
        nh = __fsqrt_rn(qh);
        nl = __fdiv_rn(fmaf(-nh, nh, qh) + ql, 2.0f * nh);
        const float ph = nh * SQRT_D_HI;
        const float pl = fmaf(nh, SQRT_D_HI, -ph) + (nh * SQRT_D_LO + nl * SQRT_D_HI);
        float dh, dl;
        fast_two_sum(ph, pl, dh, dl);
        ih = __fdiv_rn(1.0f, dh);
        const float t = fmaf(-dh, ih, 1.0f) - dl * ih;
        il = ih * t;
    }

    // exact S = H x by three exactly-transformable pieces
    float s1[4], s2[4], s3[4];
    if (amax > 0.0f) {
        const int eM = ((__float_as_int(amax) >> 23) & 0xff) - 127;
        const float q1 = __int_as_float((eM - 15 + 127) << 23);
        const float iq1 = __int_as_float((15 - eM + 127) << 23);
        const float q2 = __int_as_float((eM - 32 + 127) << 23);
        const float iq2 = __int_as_float((32 - eM + 127) << 23);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float a = rintf(x[j] * iq1) * q1;
            const float rem = x[j] - a;
            const float b = rintf(rem * iq2) * q2;
            s1[j] = a;
            s2[j] = b;
            s3[j] = rem - b;
        }
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) s1[j] = s2[j] = s3[j] = 0.0f;
    }
    wht_lane_exact(s1, lane);
    wht_lane_exact(s2, lane);
    // the third piece holds only values 2^22 and more below the row's largest
    // (almost never): skip its transform when it is zero everywhere
    if (__any_sync(FULL_MASK, s3[0] != 0.0f || s3[1] != 0.0f || s3[2] != 0.0f || s3[3] != 0.0f))
        wht_lane_exact(s3, lane);

    uint32_t part1 = 0, part2 = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float a, e1, b, e2, sh, sl;
        two_sum(s1[j], s2[j], a, e1);
        two_sum(a, s3[j], b, e2);
        fast_two_sum(b, e1 + e2, sh, sl);
        // y = S * inv
        const float yh0 = sh * ih;
        const float yl0 = fmaf(sh, ih, -yh0) + (sh * il + sl * ih);
        float yh, yl;
        fast_two_sum(yh0, yl0, yh, yl);
        const int code1 = stage_code_df<BITS, GRID>(yh, yl, tb1, tc1, p.t1, p.b1);
        const float c = __shfl_sync(FULL_MASK, tcen, code1);
        float rh, rl0, rh2, rl;
        two_sum(yh, -c, rh, rl0);
        fast_two_sum(rh, rl0 + yl, rh2, rl);
        const int code2 = stage_code_df<BITS, GRID>(rh2, rl, tb2, tc2, p.t2, p.b2);
        part1 |= (uint32_t)code1 << (j * BITS);
        part2 |= (uint32_t)code2 << (j * BITS);
    }
    // assemble words: lanes [w*LPW, (w+1)*LPW) hold word w
    const int sub = lane % LPW;
    part1 <<= sub * 4 * BITS;
    part2 <<= sub * 4 * BITS;
#pragma unroll
    for (int o = 1; o < LPW; o <<= 1) {
        part1 |= __shfl_xor_sync(FULL_MASK, part1, o);
        part2 |= __shfl_xor_sync(FULL_MASK, part2, o);
    }
    size_t drow = 0;
    if (!rvq_dst_row(p, row, drow)) return;
    if (sub == 0 && lane / LPW < W) {
        p.p1[drow * W + lane / LPW] = part1;
        p.p2[drow * W + lane / LPW] = part2;
    }
    if (lane == 0) p.norms[drow] = __fadd_rn(nh, nl);
}

// Book constants of the tensor-memory encoder's exact recompute, held in
// registers: the 32-cell stage tables (lane entries, read by shuffle; b = 4)
// and their grid maps, or the three boundaries of each stage (b = 2), and the
// stage-1 centroid of lane l & (2^b - 1).
struct FixBooks {
    float tb1, tb2, tcen;
    int tc1, tc2;
    float a1, bc1, a2, bc2;
    float b1[3], b2[3];
};

template <int MODE>
__device__ __forceinline__ FixBooks fix_books(const RvqEncodeParams &p, int lane)
{
    FixBooks f;
    f.tcen = p.c1[lane & (MODE == MODE_PAIR ? 15 : 3)];
    if constexpr (MODE == MODE_PAIR) {
        f.tb1 = p.t1.bnd[lane];
        f.tc1 = p.t1.code[lane];
        f.tb2 = p.t2.bnd[lane];
        f.tc2 = p.t2.code[lane];
        f.a1 = p.t1.a;
        f.bc1 = p.t1.bc;
        f.a2 = p.t2.a;
        f.bc2 = p.t2.bc;
    } else {
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            f.b1[k] = p.b1[k];
            f.b2[k] = p.b2[k];
        }
    }
    return f;
}

// [v > b] for the double-float v = vh + vl and an fp32 b
__device__ __forceinline__ int df_gt(float vh, float vl, float b) { return (vh > b || (vh == b && vl > 0.0f)) ? 1 : 0; }

// Boundary count of a double-float value in one stage (the tensor-memory
// encoder's books): table lookup (b = 4) or the three boundaries (b = 2).
template <int MODE>
__device__ __forceinline__ int fix_count(float vh, float vl, float tb, int tc, float a, float bc, const float (&b)[3])
{
    if constexpr (MODE == MODE_PAIR) {
        const int g = grid_cell(vh, a, bc);
        const float bnd = __shfl_sync(FULL_MASK, tb, g);
        const int cl = __shfl_sync(FULL_MASK, tc, g);
        return cl + df_gt(vh, vl, bnd);
    } else {
        return df_gt(vh, vl, b[0]) + df_gt(vh, vl, b[1]) + df_gt(vh, vl, b[2]);
    }
}

// Exact recompute of one row by one warp, for the tensor-memory encoder's
// books (symmetric b = 2, or b = 4 with grid tables): lane l holds coordinates
// 4l .. 4l + 3 (one 8-byte load).  Same arithmetic as rvq_fixup_row: S = H
// diag(s) x exactly from three pieces whose transforms are exact in fp32, Q,
// n and 1 / (n sqrt(D)) as double-floats, y = S / (n sqrt(D)) as a
// double-float, each boundary count on it; the book constants come in
// registers (no kernel-parameter reads by a runtime index).  (A variant that
// took two rows per warp, sixteen lanes each, ran slower.)  Words and norm go
// to the row's destination.
template <int MODE>
__device__ __noinline__ void rvq_fixup_tm(const RvqEncodeParams &p, int row, int lane, const FixBooks &fbm)
{
    constexpr int NR = 1;
    constexpr int BITS = MODE == MODE_PAIR ? 4 : 2;
    constexpr int W = D * BITS / 32;
    constexpr int LPR = 32 / NR, C = 4 * NR;
    constexpr int LPW = 32 / (C * BITS);  // lanes per word
    const FixBooks fb = fbm;  // to registers once (the caller's copy is in local memory)
    const int ll = lane;
    float x[C];
    {
        uint32_t w[C / 2];
#pragma unroll
        for (int k = 0; k < C / 2; ++k) w[k] = 0u;
        if (row >= 0) {
            const unsigned char *src = static_cast<const unsigned char *>(p.x) + (size_t)row * ROW_BYTES + ll * (2 * C);
            if constexpr (C == 8) {
                const uint4 u = __ldg(reinterpret_cast<const uint4 *>(src));
                w[0] = u.x; w[1] = u.y; w[2] = u.z; w[3] = u.w;
            } else {
                const uint2 u = __ldg(reinterpret_cast<const uint2 *>(src));
                w[0] = u.x; w[1] = u.y;
            }
        }
        if (p.has_sgn) {
#pragma unroll
            for (int k = 0; k < C / 2; ++k) w[k] ^= half2_sign_mask(sign_pair(p.sgn, C * ll + 2 * k));
        }
#pragma unroll
        for (int k = 0; k < C / 2; ++k) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w[k]));
            x[2 * k] = f.x;
            x[2 * k + 1] = f.y;
        }
    }
    // row max |x| and sum of squares (double-float) over the row's lanes
    float amax = 0.0f, qh = 0.0f, ql = 0.0f;
#pragma unroll
    for (int j = 0; j < C; ++j) {
        amax = fmaxf(amax, fabsf(x[j]));
        float t, e;
        two_sum(qh, x[j] * x[j], t, e);
        qh = t;
        ql += e;
    }
#pragma unroll
    for (int m = LPR / 2; m >= 1; m >>= 1) {
        amax = fmaxf(amax, __shfl_xor_sync(FULL_MASK, amax, m));
        const float oh = __shfl_xor_sync(FULL_MASK, qh, m);
        const float ol = __shfl_xor_sync(FULL_MASK, ql, m);
        float t, e;
        two_sum(qh, oh, t, e);
        e += ql + ol;
        fast_two_sum(t, e, qh, ql);
    }
    // n = sqrt(Q), den = n sqrt(D), inv = 1 / den, as double-floats
    float nh = 0.0f, nl = 0.0f, ih = 0.0f, il = 0.0f;
    if (qh > 0.0f) {
        nh = __fsqrt_rn(qh);
        nl = __fdiv_rn(fmaf(-nh, nh, qh) + ql, 2.0f * nh);
        const float ph = nh * SQRT_D_HI;
        const float pl = fmaf(nh, SQRT_D_HI, -ph) + (nh * SQRT_D_LO + nl * SQRT_D_HI);
        float dh, dl;
        fast_two_sum(ph, pl, dh, dl);
        ih = __fdiv_rn(1.0f, dh);
        const float t = fmaf(-dh, ih, 1.0f) - dl * ih;
        il = ih * t;
    }
    // exact S = H x from three pieces on the grids 2^(e-15), 2^(e-32) (e the
    // exponent of max |x|): every partial sum of up to 128 pieces is an
    // integer below 2^24 in its grid's unit
    float s1[C], s2[C], s3[C];
    {
        const int eM = amax > 0.0f ? ((__float_as_int(amax) >> 23) & 0xff) - 127 : 0;
        const float q1 = __int_as_float((eM - 15 + 127) << 23);
        const float iq1 = __int_as_float((15 - eM + 127) << 23);
        const float q2 = __int_as_float((eM - 32 + 127) << 23);
        const float iq2 = __int_as_float((32 - eM + 127) << 23);
#pragma unroll
        for (int j = 0; j < C; ++j) {
            const float a = rintf(x[j] * iq1) * q1;
            const float rem = x[j] - a;
            const float b = rintf(rem * iq2) * q2;
            s1[j] = a;
            s2[j] = b;
            s3[j] = rem - b;
        }
    }
    auto wht = [&](float (&a)[C]) {
#pragma unroll
        for (int h = 1; h < C; h <<= 1)
#pragma unroll
            for (int j = 0; j < C; ++j)
                if ((j & h) == 0) {
                    const float u = a[j], v = a[j + h];
                    a[j] = u + v;
                    a[j + h] = u - v;
                }
#pragma unroll
        for (int m = 1; m < LPR; m <<= 1) {
            const bool upper = (ll & m) != 0;
#pragma unroll
            for (int j = 0; j < C; ++j) {
                const float o = __shfl_xor_sync(FULL_MASK, a[j], m);
                a[j] = upper ? (o - a[j]) : (a[j] + o);
            }
        }
    };
    wht(s1);
    wht(s2);
    {
        bool nz = false;  // the third piece is almost always zero: skip its transform then
#pragma unroll
        for (int j = 0; j < C; ++j) nz = nz || s3[j] != 0.0f;
        if (__any_sync(FULL_MASK, nz)) wht(s3);
    }

    uint32_t part1 = 0u, part2 = 0u;
#pragma unroll
    for (int j = 0; j < C; ++j) {
        float a, e1, b, e2, sh, sl;
        two_sum(s1[j], s2[j], a, e1);
        two_sum(a, s3[j], b, e2);
        fast_two_sum(b, e1 + e2, sh, sl);
        const float yh0 = sh * ih;
        const float yl0 = fmaf(sh, ih, -yh0) + (sh * il + sl * ih);
        float yh, yl;
        fast_two_sum(yh0, yl0, yh, yl);
        const int code1 = fix_count<MODE>(yh, yl, fb.tb1, fb.tc1, fb.a1, fb.bc1, fb.b1);
        const float c = __shfl_sync(FULL_MASK, fb.tcen, code1);
        float rh, rl0, rh2, rl;
        two_sum(yh, -c, rh, rl0);
        fast_two_sum(rh, rl0 + yl, rh2, rl);
        const int code2 = fix_count<MODE>(rh2, rl, fb.tb2, fb.tc2, fb.a2, fb.bc2, fb.b2);
        part1 |= (uint32_t)code1 << (j * BITS);
        part2 |= (uint32_t)code2 << (j * BITS);
    }
    // words: lanes [w LPW, (w + 1) LPW) of a row hold word w
    const int sub = ll % LPW;
    part1 <<= sub * C * BITS;
    part2 <<= sub * C * BITS;
#pragma unroll
    for (int o = 1; o < LPW; o <<= 1) {
        part1 |= __shfl_xor_sync(FULL_MASK, part1, o);
        part2 |= __shfl_xor_sync(FULL_MASK, part2, o);
    }
    size_t drow = 0;
    if (row < 0 || !rvq_dst_row(p, row, drow)) return;
    if (sub == 0) {
        p.p1[drow * W + ll / LPW] = part1;
        p.p2[drow * W + ll / LPW] = part2;
    }
    if (ll == 0) p.norms[drow] = __fadd_rn(nh, nl);
}

// The tensor-memory encoder's exact recompute of one row: b = 2 books by
// rvq_fixup_tm; b = 4 by rvq_fixup_row (the grid tables read in place), which
// measured a few per cent faster there.
template <int MODE>
__device__ __forceinline__ void fixup_one(const RvqEncodeParams &p, int row, int lane, const FixBooks &fb)
{
    if constexpr (MODE == MODE_PAIR)
        rvq_fixup_row<4, true, 0>(p, nullptr, 0, row, lane, fb.tb1, fb.tc1, fb.tb2, fb.tc2, fb.tcen);
    else
        rvq_fixup_tm<MODE>(p, row, lane, fb);
}

// SGN: the randomised-sign rotation (a separate instantiation, so that the
// plain rotation carries no per-row test).
template <int BITS, int MODE, bool SGN>
__device__ __forceinline__ void rvq_encode_body(const RvqEncodeParams &p, int cta, int ncta)
{
    constexpr bool GRID = MODE == MODE_GRID;
    constexpr int L = 1 << BITS;
    constexpr int E = 32 / BITS;
    constexpr int W = D * BITS / 32;
    constexpr int WL = W / 2;  // words of a half row
    constexpr int WARPS = enc_warps(BITS, MODE);
    constexpr bool ROLLED = MODE == MODE_GRID || MODE == MODE_PLAIN;
    constexpr int PP = enc_pairs(BITS);
    static_assert(!(MODE == MODE_SYM && BITS == 2), "symmetric b = 2 books: rvq_encode_tm_body");
    static_assert(MODE != MODE_PAIR, "the b = 4 pair table: rvq_encode_tm_body");
    extern __shared__ __align__(128) unsigned char smem_raw[];
    unsigned char *stab = smem_1k(smem_raw);       // cell tables (GRID)
    uint4 *ssg = reinterpret_cast<uint4 *>(stab + enc_tab_bytes(MODE));  // sign masks
    unsigned char *smem = stab + enc_tab_bytes(MODE) + ENC_SGN_BYTES;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int rr = lane & 15, hh = lane >> 4;
    unsigned char *ring = smem + warp * (ENC_STAGES * ENC_BLOCK);
    unsigned char *wextra = smem + WARPS * ENC_STAGES * ENC_BLOCK + warp * (enc_warp_bytes(BITS, MODE) - ENC_STAGES * (ENC_BLOCK + 8));
    float2 *yp = reinterpret_cast<float2 *>(wextra);                                   // ROLLED only
    uint32_t *ws = reinterpret_cast<uint32_t *>(wextra + PP * 32 * 8) + lane * 2 * (WL + 1);  // ROLLED only
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + WARPS * (enc_warp_bytes(BITS, MODE) - ENC_STAGES * 8)) +
                     warp * ENC_STAGES;

    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < ENC_STAGES; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    __syncwarp();

    const uint64_t pol = l2_policy_evict_first();
    const float tb1 = p.t1.bnd[lane];
    const int tc1 = p.t1.code[lane];
    const float tb2 = p.t2.bnd[lane];
    const int tc2 = p.t2.code[lane];
    const float tcen = p.c1[lane & (L - 1)];
    if constexpr (GRID) {
        // cell tables, replicated per lane; an empty cell (boundary -inf)
        // always takes code + 1, so its centroid step is 0
        float4 *t1s = reinterpret_cast<float4 *>(stab);
        float2 *t2s = reinterpret_cast<float2 *>(stab + 32 * 32 * 16);
        for (int i = threadIdx.x; i < 32 * 32; i += blockDim.x) {
            const int g = i >> 5;
            const int c = p.t1.code[g];
            const bool empty = !(p.t1.bnd[g] > -3.0e38f);
            const float chi = p.c1[c + 1];
            const float clo = p.c1[empty ? c + 1 : c];
            t1s[i] = make_float4(p.t1.bnd[g], __int_as_float(c), clo, chi - clo);
            t2s[i] = make_float2(p.t2.bnd[g], __int_as_float(p.t2.code[g]));
        }
        __syncthreads();
    }
    if (threadIdx.x < 16) {
        // chunk t & 7 (8 coordinates) of half t >> 3: coordinates 64 (t >> 3) + 8 (t & 7) ..
        const int c0 = 64 * (threadIdx.x >> 3) + 8 * (threadIdx.x & 7);
        ssg[threadIdx.x] = make_uint4(half2_sign_mask(sign_pair(p.sgn, c0)), half2_sign_mask(sign_pair(p.sgn, c0 + 2)),
                                      half2_sign_mask(sign_pair(p.sgn, c0 + 4)), half2_sign_mask(sign_pair(p.sgn, c0 + 6)));
    }
    __syncthreads();
    // this lane's table columns: entry g at g * 512 (stage 1) / g * 256 (stage 2)
    const unsigned char *t1l = stab + lane * 16;
    const unsigned char *t2l = stab + 32 * 32 * 16 + lane * 8;
    const int nblk = (p.N + ER - 1) / ER;
    const int gw = cta * WARPS + warp;
    const int tw = ncta * WARPS;

    auto issue = [&](int blk, int s) {
        if (lane == 0) {
            mbar_arrive_expect_tx(&bars[s], (uint32_t)ENC_BLOCK);
            tma_load_2d(ring + s * ENC_BLOCK, &p.tmap, 0, blk * ER, &bars[s], pol);
            tma_load_2d(ring + s * ENC_BLOCK + ENC_BLOCK / 2, &p.tmap, 64, blk * ER, &bars[s], pol);
        }
    };
#pragma unroll
    for (int s = 0; s < ENC_STAGES; ++s) {
        const int blk = gw + s * tw;
        if (blk < nblk) issue(blk, s);
    }

    for (int it = 0;; ++it) {
        const int blk = gw + it * tw;
        if (blk >= nblk) break;
        const int s = it % ENC_STAGES;
        const bool ok = mbar_wait_bounded(&bars[s], (uint32_t)(it / ENC_STAGES) & 1u);
        if (!__all_sync(FULL_MASK, ok)) {
            // A copy never landed: record it, wait (bounded) for the other
            // copies this warp has in flight so none writes into a retired
            // buffer, and stop.
            if (lane == 0) atomicOr(&VQ_RVQ_ERR, (unsigned)VQ_DEVERR_WAIT_TIMEOUT);
            for (int k = 1; k < ENC_STAGES; ++k) {
                const int it2 = it + k;
                if (gw + it2 * tw < nblk)
                    (void)mbar_wait_bounded(&bars[it2 % ENC_STAGES], (uint32_t)(it2 / ENC_STAGES) & 1u);
            }
            return;
        }
        const unsigned char *sbuf = ring + s * ENC_BLOCK;
        const int row = blk * ER + rr;
        const bool valid = row < p.N;

        // ---- this thread's input half x_h = x[64h .. 64h + 63] as pairs
        // (x_h[k], x_h[k + 32]); the bit-5 butterfly runs on the fp16 values
        // (only the second operand is converted, the first is added as an
        // fp16 operand), then bits 0-4 across the array: Z_h = H64 x_h.
        float2 v[32];
        {
            const unsigned char *src = sbuf + hh * (ENC_BLOCK / 2);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint4 la = *reinterpret_cast<const uint4 *>(src + swz128(rr, c));
                uint4 lb = *reinterpret_cast<const uint4 *>(src + swz128(rr, c + 4));
                if constexpr (SGN) {
                    // randomised signs: x -> diag(s) x on the fp16 bits
                    const uint4 ma = ssg[hh * 8 + c], mb = ssg[hh * 8 + c + 4];
                    la = make_uint4(la.x ^ ma.x, la.y ^ ma.y, la.z ^ ma.z, la.w ^ ma.w);
                    lb = make_uint4(lb.x ^ mb.x, lb.y ^ mb.y, lb.z ^ mb.z, lb.w ^ mb.w);
                }
                const __half *pa = reinterpret_cast<const __half *>(&la);
                const __half *pb = reinterpret_cast<const __half *>(&lb);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float b = __half2float(pb[j]);
                    v[8 * c + j] = make_float2(add_f16_f32(pa[j], b), add_f16_f32(pa[j], -b));
                }
            }
        }

        // ---- norm: the sums of squares after that stage add up to twice sum x^2
        float2 acc[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i] = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int k = 0; k < 32; ++k) acc[k & 3] = __ffma2_rn(v[k], v[k], acc[k & 3]);
        acc[0] = __fadd2_rn(acc[0], acc[2]);
        acc[1] = __fadd2_rn(acc[1], acc[3]);
        acc[0] = __fadd2_rn(acc[0], acc[1]);
        const float qs = acc[0].x + acc[0].y;
        const float q = 0.5f * (qs + __shfl_xor_sync(FULL_MASK, qs, 16));
        const float n = __fsqrt_rn(q);
        const float den = n * SQRT_D_HI;
        if constexpr (MODE != MODE_SYM) {
            // table and plain modes quantize y = S / den
            const float inv = q > 0.0f ? __frcp_rn(den) : 0.0f;
            const float2 inv2 = make_float2(inv, inv);
#pragma unroll
            for (int k = 0; k < 32; ++k) v[k] = __fmul2_rn(v[k], inv2);
        }
        const float2 neg1 = make_float2(-1.0f, -1.0f);
#pragma unroll
        for (int h = 1; h < 32; h <<= 1) {
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                if ((k & h) == 0) {
                    const float2 a = v[k], b = v[k + h];
                    v[k] = __fadd2_rn(a, b);
                    v[k + h] = __ffma2_rn(b, neg1, a);
                }
            }
        }
        // ---- bit 6 across the two threads: y_0 = Z_0 + Z_1, y_1 = Z_0 - Z_1;
        // afterwards v[k] = (y_h[k], y_h[k + 32]) of this thread's output half
        {
            const float2 sgn = hh ? neg1 : make_float2(1.0f, 1.0f);
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                const float2 o = make_float2(__shfl_xor_sync(FULL_MASK, v[k].x, 16),
                                             __shfl_xor_sync(FULL_MASK, v[k].y, 16));
                v[k] = __ffma2_rn(v[k], sgn, o);
            }
        }

        // symmetric modes quantize S itself against thresholds scaled by den
        SymRow sk;
        sk.bb = p.b1[(1 << BITS) - 2] * den;
        sk.be = p.b2[(1 << BITS) - 2] * den;
        sk.bc2 = (p.b1[(1 << BITS) - 2] - p.c1[(1 << BITS) - 2]) * den;
        sk.dc = (p.c1[(1 << BITS) - 1] - p.c1[(1 << BITS) - 2]) * den;
        sk.c1 = p.c1[(1 << BITS) - 1] * den;
        sk.k1 = sk.k2 = sk.G1 = sk.G2 = 0.0f;
        const float guard = MODE == MODE_SYM ? p.guard * den : p.guard;

        // ---- two-stage boundary count and LSB-first packing: word kx of the
        // half from the first coordinates of pairs [kx*E, kx*E + E), word
        // kx + WL/2 from the second ones.
        float mx = __int_as_float(0x7f800000), my = mx;
        uint32_t wa1[WL], wa2[WL];
        if constexpr (!ROLLED) {
            // symmetric 1/2-bit books: unrolled, in registers
#pragma unroll
            for (int kx = 0; kx < WL / 2; ++kx) {
                uint32_t a1x = 0u, a2x = 0u, a1y = 0u, a2y = 0u;
#pragma unroll
                for (int i = E - 1; i >= 0; --i) {
                    const float2 y2 = v[kx * E + i];
                    sym1_code(y2.x, sk, a1x, a2x, mx);
                    sym1_code(y2.y, sk, a1y, a2y, my);
                }
                wa1[kx] = ~a1x;
                wa2[kx] = ~a2x;
                wa1[WL / 2 + kx] = ~a1y;
                wa2[WL / 2 + kx] = ~a2y;
            }
        } else {
            // table / plain count: slices of PP pairs through the scratch
            // yp[i * 32 + lane], a rolled word loop, words staged per lane
#pragma unroll 1
            for (int ps = 0; ps < 32 / PP; ++ps) {
#pragma unroll
                for (int q4 = 0; q4 < 32 / PP; ++q4) {
                    if (ps == q4) {
#pragma unroll
                        for (int i = 0; i < PP; ++i) yp[i * 32 + lane] = v[q4 * PP + i];
                    }
                }
#pragma unroll 1
                for (int w = 0; w < PP / E; ++w) {
                    uint32_t a1x = 0u, a2x = 0u, a1y = 0u, a2y = 0u;
#pragma unroll
                    for (int i = 0; i < E; ++i) {
                        const float2 y2 = yp[(w * E + i) * 32 + lane];
                        int cx1, cy1, cx2, cy2;
                        if constexpr (GRID) {
                            grid2_code(y2.x, p.t1, p.t2, t1l, t2l, cx1, cx2, mx);
                            grid2_code(y2.y, p.t1, p.t2, t1l, t2l, cy1, cy2, my);
                        } else {
                            cx1 = stage_code<BITS, GRID>(y2.x, tb1, tc1, p.t1, p.b1, mx);
                            cy1 = stage_code<BITS, GRID>(y2.y, tb1, tc1, p.t1, p.b1, my);
                            const float rx = y2.x - __shfl_sync(FULL_MASK, tcen, cx1);
                            const float ry = y2.y - __shfl_sync(FULL_MASK, tcen, cy1);
                            cx2 = stage_code<BITS, GRID>(rx, tb2, tc2, p.t2, p.b2, mx);
                            cy2 = stage_code<BITS, GRID>(ry, tb2, tc2, p.t2, p.b2, my);
                        }
                        a1x = __funnelshift_r(a1x, (uint32_t)cx1, BITS);
                        a2x = __funnelshift_r(a2x, (uint32_t)cx2, BITS);
                        a1y = __funnelshift_r(a1y, (uint32_t)cy1, BITS);
                        a2y = __funnelshift_r(a2y, (uint32_t)cy2, BITS);
                    }
                    const int kx = ps * (PP / E) + w;
                    ws[kx] = a1x;
                    ws[WL / 2 + kx] = a1y;
                    ws[WL + 1 + kx] = a2x;
                    ws[WL + 1 + WL / 2 + kx] = a2y;
                }
            }
#pragma unroll
            for (int i = 0; i < WL; ++i) {
                wa1[i] = ws[i];
                wa2[i] = ws[WL + 1 + i];
            }
        }
        const float m = fminf(mx, my);
        // a zero row has no direction: always take the exact path for it
        const bool hflag = valid && (!(m >= guard) || !(q > 0.0f));
        // (the shuffle runs on every lane: no short-circuit around it)
        const int pflag = __shfl_xor_sync(FULL_MASK, hflag ? 1 : 0, 16);
        const bool flag = hflag || pflag != 0;

        // ---- the fast words of this half, straight to global memory (the 16
        // rows x 2 halves of a block are contiguous there); rows with a value
        // inside the guard band are written by the exact recompute instead
        size_t drow = 0;
        const bool okrow = valid && !flag && rvq_dst_row(p, row, drow);
        if (okrow) {
            uint32_t *d1 = p.p1 + drow * W + hh * WL;
            uint32_t *d2 = p.p2 + drow * W + hh * WL;
            if constexpr (WL == 2) {
                *reinterpret_cast<uint2 *>(d1) = make_uint2(wa1[0], wa1[1]);
                *reinterpret_cast<uint2 *>(d2) = make_uint2(wa2[0], wa2[1]);
            } else {
#pragma unroll
                for (int i = 0; i < WL / 4; ++i) {
                    reinterpret_cast<uint4 *>(d1)[i] = make_uint4(wa1[4 * i], wa1[4 * i + 1], wa1[4 * i + 2], wa1[4 * i + 3]);
                    reinterpret_cast<uint4 *>(d2)[i] = make_uint4(wa2[4 * i], wa2[4 * i + 1], wa2[4 * i + 2], wa2[4 * i + 3]);
                }
            }
            if (hh == 0) p.norms[drow] = n;
        }

        // ---- rows with a value inside the guard band: exact recompute by the warp
        unsigned fl = __ballot_sync(FULL_MASK, flag) & 0xffffu;
        while (fl) {
            const int r = __ffs(fl) - 1;
            fl &= fl - 1;
            rvq_fixup_row<BITS, GRID>(p, sbuf, r, blk * ER + r, lane, tb1, tc1, tb2, tc2, tcen);
        }
        __syncwarp();

        // ---- recycle this stage for the block ENC_STAGES iterations ahead
        fence_proxy_async_smem();
        {
            const int nb = blk + ENC_STAGES * tw;
            if (nb < nblk) issue(nb, s);
        }

    }
}

// ------------------------------------------- the library's books: shared pieces
//
// The pair table of the b = 4 books lives in shared memory replicated
// P4_REP = 16 times (cell g, replica j at byte (16 g + j) 8) and lane l reads
// replica l & 15: an 8-byte read is served per half-warp, so the 16 lanes of
// each half always hit 16 distinct bank pairs and the lookup is free of bank
// conflicts.  The quantizers work on S = H x directly: with den = n sqrt(D),
// y > bnd exactly when bnd den - S is negative (one FMA rounding of an exact
// product-difference), the cell coordinate is fma(S, a / den, bc) and the
// margin |bnd den - S| is compared with guard den; the host builds the table
// with every step at least three guard bands inside its cell, which absorbs
// the rounding of a / den (the cell a value lands in can differ from the
// y-domain map only near cell edges, where the neighbouring cell's entry
// gives the same pair).
constexpr int P4_REP = 16;
constexpr int P4_TAB_BYTES = PT_CELLS * P4_REP * 8;

// Per-row constants of the symmetric b = 2 quantizer (units of S = H x).
__device__ __forceinline__ SymRow sym2_row(float den, float g, float b1u, float b2u, float bc2u, float dcu,
                                           float kb1, float kb2)
{
    SymRow k;
    k.bb = b1u * den;
    k.be = b2u * den;
    k.bc2 = bc2u * den;
    k.dc = dcu * den;
    k.c1 = 0.0f;
    // approximate reciprocal (a zero row gives inf here; it always takes the
    // exact path)
    float rden;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(rden) : "f"(den));
    k.k1 = kb1 * rden;
    k.k2 = kb2 * rden;
    k.G1 = g * (k.bb + 2.0f * g);
    k.G2 = g * (k.be + 2.0f * g);
    return k;
}

// Both 4-bit codes of the coordinate S (pair i1 | i2 << 4 in the low byte).
// tab: this lane's replica as a 32-bit shared address, less the magic
// constant's bits shifted by 7, so that the cell's entry is at tab + (gb << 7)
// with gb the bits of the cell FMA (0x4B400000 + cell).
__device__ __forceinline__ uint32_t pair_code_s(float s, float a, float bc, float den, uint32_t tab, float &m)
{
    const float u = __saturatef(fmaf(s, a, bc));
    // cell in [0, PT_CELLS - 1]: u is saturated (NaN saturates to 0)
    const uint32_t gb = __float_as_uint(fmaf(u, (float)(PT_CELLS - 1), GRID_MAGIC));
    uint32_t ex, ey;
    asm("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(ex), "=r"(ey) : "r"(tab + (gb << 7)));
    // S > bnd den exactly when d is negative (an exact tie gives +0)
    const float d = fmaf(__uint_as_float(ex), den, -s);
    m = fminf(m, fabsf(d));
    return __byte_perm(ey, 0u, __float_as_uint(d) >> 31);
}

// ------------------------------------------- encode on the 5th-generation tensor cores
//
// The library's books (symmetric b = 2, and b = 4 with a pair table), 128 rows
// per tile: the whole rotation S = X H128 is one D = X B^T of M = N = K = 128
// (eight tcgen05.mma of K = 16, fp16 operands - the products x_d (+-1) are
// exact - fp32 accumulation) into tensor memory; B = H128 diag(s) (the
// randomised signs, when given, ride in B for free) is built once per CTA in
// the K-major 128-byte-swizzled layout the X tiles arrive in by TMA.  Then a
// thread owns a row: it takes the norm from its fp16 row in the staged tile
// (exact squares by mixed-precision FMAs), reads its 128 accumulators
// (tcgen05.ld, tensor-memory lane = row), quantizes its coordinates in
// natural order and stores whole words; no butterflies,
// no operand permutes, no cross-lane packing.  Roles (one persistent CTA per
// SM): warp 0 streams X tiles (TMA, TE_STAGES-deep ring), warp 1 owns the
// tensor memory and issues the MMAs (one thread), TE_G groups of four warps
// run the epilogue on alternate tiles, each group with its own accumulator
// buffer (128 columns), and TE_FIX warps recompute flagged rows.  A row with
// a value inside the guard band is queued (its global index, in a shared-memory
// list) for the fixup warps, which redo it exactly (rvq_fixup_row, the row
// read again from global memory) off the epilogue's critical path: an epilogue
// warp that stopped for a recompute would hold its accumulator buffer and,
// through the in-order MMA issue, the whole pipeline.  When the list is full
// the epilogue warp recomputes the row itself.
// Every wait is bounded; on a timeout the CTA records VQ_DEVERR_WAIT_TIMEOUT,
// waits (bounded) for its copies in flight, frees its tensor memory and
// returns.
// Sum of the squares of the 8 fp16 values of a 16-byte chunk: each square
// exact (fp16 operands, fp32 result of a mixed-precision FMA), 8 fp32 sums.
__device__ __forceinline__ float sq8_f16(uint4 v)
{
    float a = 0.0f;
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const unsigned short lo = (unsigned short)(w[j] & 0xffffu), hi = (unsigned short)(w[j] >> 16);
        asm("fma.rn.f32.f16 %0, %1, %1, %0;" : "+f"(a) : "h"(lo));
        asm("fma.rn.f32.f16 %0, %1, %1, %0;" : "+f"(a) : "h"(hi));
    }
    return a;
}

constexpr int TE_M = 128;
constexpr int TE_G = 3;                       // epilogue groups (4 warps each)
constexpr int TE_FIX = 2;                     // fixup warps
constexpr int TE_FIX0 = 2 + 4 * TE_G;         // first fixup warp
constexpr int TE_THREADS = 32 * (TE_FIX0 + TE_FIX);
constexpr int TE_FQ = 1024;                   // flagged-row list entries per CTA

constexpr int TE_HALF = TE_M * 128;           // a 64-coordinate half of a tile (16 KB)
constexpr int TE_TILE = 2 * TE_HALF;          // 32 KB
constexpr int TE_BOP = 2 * 128 * 128;         // B = H128 diag(s), fp16, 32 KB
__host__ __device__ constexpr int te_stages(int mode) { return mode == MODE_PAIR ? 3 : 4; }
__host__ __device__ constexpr int te_smem(int mode)
{
    return 1024 + TE_BOP + (mode == MODE_PAIR ? P4_TAB_BYTES : 0) + te_stages(mode) * TE_TILE + 256 + 4 * TE_FQ + 32;
}
static_assert(te_smem(MODE_PAIR) <= SMEM_MAX && te_smem(MODE_SYM) <= SMEM_MAX, "tensor-memory encoder shared memory");

template <int MODE>
__device__ __forceinline__ void rvq_encode_tm_body(const RvqEncodeParams &p, int cta, int ncta)
{
    constexpr int BITS = MODE == MODE_PAIR ? 4 : 2;
    constexpr int W = D * BITS / 32;  // words per row and stream
    constexpr int NST = te_stages(MODE);
    extern __shared__ __align__(128) unsigned char smem_raw[];
    unsigned char *base = smem_1k(smem_raw);
    unsigned char *bop = base;                                    // B: half h at h * 16 KB
    uint2 *ptab = reinterpret_cast<uint2 *>(base + TE_BOP);       // MODE_PAIR only
    unsigned char *ring = base + TE_BOP + (MODE == MODE_PAIR ? P4_TAB_BYTES : 0);
    uint64_t *bars = reinterpret_cast<uint64_t *>(ring + NST * TE_TILE);
    uint64_t *x_full = bars, *x_empty = bars + NST;
    uint64_t *acc_full = bars + 2 * NST, *acc_empty = acc_full + TE_G;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(acc_empty + TE_G);
    volatile uint32_t *abort_flag = tslot + 1;
    // flagged-row list: entries written, entries claimed by the fixup warps,
    // epilogue warps done, the entries (global row + 1; 0 = not yet written)
    uint32_t *fq_n = tslot + 2, *fq_take = tslot + 3, *fq_done = tslot + 4;
    volatile uint32_t *fq = tslot + 8;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ntiles = (p.N + TE_M - 1) / TE_M;

    // The b = 4 pair table, replicated P4_REP times (entry i a copy of cell
    // i / P4_REP): its cells are read first thing, before the tile loads
    // crowd the memory system, from device memory when the host placed them
    // there (else from the kernel parameters, slower at per-thread
    // addresses), all of a thread's reads before its stores; the stores
    // follow the first barrier and the set-up's last barrier covers them.
    constexpr int NPT = MODE == MODE_PAIR ? (PT_CELLS * P4_REP + TE_THREADS - 1) / TE_THREADS : 1;
    [[maybe_unused]] uint2 cell[NPT];
    if constexpr (MODE == MODE_PAIR) {
        static_assert((PT_CELLS * P4_REP) % TE_THREADS == 0, "whole rounds of the table copy");
        if (p.pt_dev != nullptr) {
#pragma unroll
            for (int k = 0; k < NPT; ++k) cell[k] = __ldg(p.pt_dev + (threadIdx.x + k * TE_THREADS) / P4_REP);
        } else {
#pragma unroll
            for (int k = 0; k < NPT; ++k) cell[k] = p.pt.ent[(threadIdx.x + k * TE_THREADS) / P4_REP];
        }
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(&x_full[s], 1);
            mbar_init(&x_empty[s], 4);
        }
        for (int g = 0; g < TE_G; ++g) {
            mbar_init(&acc_full[g], 1);
            mbar_init(&acc_empty[g], 4);
        }
        *abort_flag = 0u;
        *fq_n = 0u;
        *fq_take = 0u;
        *fq_done = 0u;
        fence_mbar_init();
    }
    __syncthreads();
    // the producer's first tiles go out now, under the rest of the set-up
    const uint64_t pol = l2_policy_evict_first();
    auto load_tile = [&](int t, int s) {
        unsigned char *dst = ring + s * TE_TILE;
        mbar_arrive_expect_tx(&x_full[s], (uint32_t)TE_TILE);
        tma_load_2d(dst, &p.tmap, 0, t * TE_M, &x_full[s], pol);
        tma_load_2d(dst + TE_HALF, &p.tmap, 64, t * TE_M, &x_full[s], pol);
    };
    if (threadIdx.x == 0)
        for (int s = 0; s < NST && cta + s * ncta < ntiles; ++s) load_tile(cta + s * ncta, s);
    if constexpr (MODE == MODE_PAIR) {
#pragma unroll
        for (int k = 0; k < NPT; ++k) ptab[threadIdx.x + k * TE_THREADS] = cell[k];
    }
    for (int i = threadIdx.x; i < TE_FQ; i += blockDim.x) fq[i] = 0u;
    // B[n][k] = H128[j(n)][k] s_k, fp16, K-major with the 128-byte swizzle:
    // 16-byte chunk c (k = 8c .. 8c + 7) of row n.  Row n of B is column n of
    // the accumulator; for the symmetric books the output coordinates are
    // interleaved so that a thread's registers 2b and 2b + 1 of a 32-column
    // load are coordinates 32q + b and 32q + 16 + b (the two words the
    // quantizer fills side by side, as one fp32 pair): j(32q + 2b + e) =
    // 32q + 16e + b.  The b = 4 quantizer works per coordinate: j(n) = n.
    for (int i = threadIdx.x; i < 128 * 16; i += blockDim.x) {
        const int n = i >> 4, c = i & 15;
        const int j = MODE == MODE_SYM ? (n & ~31) + 16 * (n & 1) + ((n & 31) >> 1) : n;
        uint32_t h[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int k0 = 8 * c + 2 * e;
            const uint32_t lo = ((__popc(j & k0) & 1) ? 0xBC00u : 0x3C00u) ^ (p.has_sgn ? (((p.sgn[k0 >> 5] >> (k0 & 31)) & 1u) << 15) : 0u);
            const uint32_t hi = ((__popc(j & (k0 + 1)) & 1) ? 0xBC00u : 0x3C00u) ^
                                (p.has_sgn ? (((p.sgn[(k0 + 1) >> 5] >> ((k0 + 1) & 31)) & 1u) << 15) : 0u);
            h[e] = lo | (hi << 16);
        }
        *reinterpret_cast<uint4 *>(bop + (c >> 3) * TE_HALF + swz128(n, c & 7)) = make_uint4(h[0], h[1], h[2], h[3]);
    }
    fence_proxy_async_smem();  // B is read by the MMAs (async proxy)
    if (warp == 1) tmem_alloc(tslot, 512);
    qt_fence_before();
    __syncthreads();
    qt_fence_after();
    const uint32_t tmem = *tslot;

    // Exact recomputes from the flagged-row list: the calling warp claims the
    // next entry until the list ends (every epilogue warp done and no entry
    // left).  The fixup warps run this from the start, the epilogue warps
    // once their tiles are done (so that a list still full at the end drains
    // on all of them).
    auto drain = [&](const FixBooks &fb) {
        for (;;) {
            uint32_t k = 0u;
            if (lane == 0) k = atomicAdd(fq_take, 1u);
            k = __shfl_sync(FULL_MASK, k, 0);
            if (k >= (uint32_t)TE_FQ) break;
            // wait for entry k, or for every epilogue warp to finish with fewer entries
            uint32_t e = 0u;
            bool ok = true;
            const uint64_t t0 = globaltimer_ns();
            for (;;) {
                e = fq[k];
                if (e != 0u) break;
                if (*reinterpret_cast<volatile uint32_t *>(fq_done) == 4u * TE_G) {
                    __threadfence_block();
                    e = fq[k];
                    if (e != 0u || *reinterpret_cast<volatile uint32_t *>(fq_n) <= k) break;
                }
                if (globaltimer_ns() - t0 > MBAR_TIMEOUT_NS) {
                    ok = false;
                    break;
                }
                __nanosleep(256);
            }
            e = __shfl_sync(FULL_MASK, e, 0);
            if (!__all_sync(FULL_MASK, ok)) {
                if (lane == 0) atomicOr(&VQ_RVQ_ERR, (unsigned)VQ_DEVERR_WAIT_TIMEOUT);
                break;
            }
            if (e == 0u) break;  // the list ended before entry k
            __threadfence_block();
            fixup_one<MODE>(p, (int)(e - 1u), lane, fb);
        }
    };

    if (warp == 0) {
        // ---- producer (tiles 0 .. NST - 1 went out during the set-up)
        if (lane == 0) {
            int i = 0;
            for (int t = cta; t < ntiles; t += ncta, ++i) {
                if (i < NST) continue;
                const int s = i % NST;
                if (!mbar_wait_bounded(&x_empty[s], (uint32_t)((i / NST) - 1) & 1u)) {
                    atomicOr(&VQ_RVQ_ERR, (unsigned)VQ_DEVERR_WAIT_TIMEOUT);
                    *abort_flag = 1u;
                    break;
                }
                if (*abort_flag) break;
                load_tile(t, s);
            }
            for (int k = 0; k < NST && k < i; ++k) {
                const int j = i - 1 - k;
                (void)mbar_wait_bounded(&x_full[j % NST], (uint32_t)(j / NST) & 1u);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---- MMA issue: tile i into accumulator buffer i % TE_G
        if (lane == 0) {
            constexpr uint32_t IDESC = qt_idesc(128);
            const uint32_t bb = smem_u32(bop), rb = smem_u32(ring);
            int i = 0;
            for (int t = cta; t < ntiles; t += ncta, ++i) {
                const int s = i % NST, a = i % TE_G;
                bool ok = mbar_wait_bounded(&x_full[s], (uint32_t)(i / NST) & 1u);
                if (ok && i >= TE_G) ok = mbar_wait_bounded(&acc_empty[a], (uint32_t)((i / TE_G) - 1) & 1u);
                if (!ok || *abort_flag) {
                    if (!ok) atomicOr(&VQ_RVQ_ERR, (unsigned)VQ_DEVERR_WAIT_TIMEOUT);
                    *abort_flag = 1u;
                    break;
                }
                qt_fence_after();
                const uint32_t xa = rb + s * TE_TILE;
#pragma unroll
                for (int kb = 0; kb < 2; ++kb) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        qt_mma(tmem + (uint32_t)(a * 128), qt_desc(xa + kb * TE_HALF + kk * 32),
                               qt_desc(bb + kb * TE_HALF + kk * 32), IDESC, (kb | kk) ? 1u : 0u);
                }
                qt_commit(&acc_full[a]);
            }
        }
        __syncwarp();
    } else if (warp < TE_FIX0) {
        // ---- epilogue group g: tiles i with i % TE_G == g; thread = row
        const int g = (warp - 2) >> 2;
        const int q = warp & 3;  // tensor-memory lane quadrant of this warp
        const int r = 32 * q + lane;
        const uint32_t tl = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(g * 128);
        const FixBooks fb = fix_books<MODE>(p, lane);  // exact recompute
        [[maybe_unused]] const float b1u = p.b1[2], b2u = p.b2[2];
        [[maybe_unused]] const float bc2u = p.b1[2] - p.c1[2], dcu = p.c1[3] - p.c1[2];
        [[maybe_unused]] const float kb1 = __fdiv_rn(2.0f, b1u), kb2 = __fdiv_rn(2.0f, b2u);
        [[maybe_unused]] const float pa = p.pt.a, pbc = p.pt.bc;
        [[maybe_unused]] const uint32_t tab =
            smem_u32(ptab) + 8u * (uint32_t)(lane & (P4_REP - 1)) - (0x4B400000u << 7);
        const bool dense = p.dst_off == nullptr && p.S_dst == p.S && p.S_q == p.S;
        int i = 0;
        for (int t = cta; t < ntiles; t += ncta, ++i) {
            if (i % TE_G != g) continue;
            const int s = i % NST;
            const bool ok = mbar_wait_bounded(&acc_full[g], (uint32_t)(i / TE_G) & 1u);
            if (!__all_sync(FULL_MASK, ok) || *abort_flag) {
                if (!ok && lane == 0) atomicOr(&VQ_RVQ_ERR, (unsigned)VQ_DEVERR_WAIT_TIMEOUT);
                *abort_flag = 1u;
                break;
            }
            qt_fence_after();
            const int row = t * TE_M + r;
            const bool valid = row < p.N;

            // the norm from the row's fp16 values in the staged tile: exact
            // squares (fp16 operands, fp32 result), fp32 sums in 16 partial
            // sums of 8 (12 roundings deep at most)
            const unsigned char *xt = ring + s * TE_TILE;
            float ps[16];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 v = *reinterpret_cast<const uint4 *>(xt + h * TE_HALF + swz128(r, c));
                    ps[8 * h + c] = sq8_f16(v);
                }
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) ps[k] += ps[k + 8];
#pragma unroll
            for (int k = 0; k < 4; ++k) ps[k] += ps[k + 4];
            ps[0] += ps[2];
            ps[1] += ps[3];
            const float qn = ps[0] + ps[1];
            const float n = __fsqrt_rn(qn);
            const float den = n * SQRT_D_HI;
            // the staged tile has been read (the MMAs are done with it too):
            // free the stage now, so that the producer keeps the ring full
            // through the quantization (a flagged row is re-read from global
            // memory by the exact recompute)
            __syncwarp();
            if (lane == 0) mbar_arrive(&x_empty[s]);

            // pass 2: quantize the row in natural coordinate order, 32
            // coordinates (one tensor-memory load) at a time, the next load in
            // flight during each chunk; the words go straight to the row's
            // destination (a flagged row is rewritten by the exact recompute)
            size_t drow = (size_t)row;
            const bool okrow = valid && (dense || rvq_dst_row(p, row, drow));
            uint32_t *d1 = p.p1 + drow * W, *d2 = p.p2 + drow * W;
            uint32_t va[32], vb[32];
            bool flag;
            if constexpr (MODE == MODE_SYM) {
                const SymRow sk = sym2_row(den, p.guard * den, b1u, b2u, bc2u, dcu, kb1, kb2);
                float m1 = __int_as_float(0x7f800000), m2 = m1;
                // words 2c (coordinates 32c .. 32c + 15) and 2c + 1, code j at bits 2j
                auto chunk = [&](const uint32_t (&v)[32], int c) {
                    uint32_t a1x = 0u, a2x = 0u, a1y = 0u, a2y = 0u;
#pragma unroll
                    for (int b = 15; b >= 0; --b)
                        sym2_code2(make_float2(__uint_as_float(v[2 * b]), __uint_as_float(v[2 * b + 1])), sk, a1x, a2x,
                                   a1y, a2y, m1, m2);
                    uint32_t x1, x2, y1, y2;
                    sym2_words(a1x, a2x, x1, x2);
                    sym2_words(a1y, a2y, y1, y2);
                    if (okrow) {
                        *reinterpret_cast<uint2 *>(d1 + 2 * c) = make_uint2(x1, y1);
                        *reinterpret_cast<uint2 *>(d2 + 2 * c) = make_uint2(x2, y2);
                    }
                };
                qt_ld32(tl, va);
#pragma unroll 1
                for (int c = 0; c < 4; c += 2) {
                    qt_wait_ld();
                    qt_hold(va);
                    qt_ld32(tl + 32 * (c + 1), vb);
                    chunk(va, c);
                    qt_wait_ld();
                    qt_hold(vb);
                    if (c + 2 < 4) qt_ld32(tl + 32 * (c + 2), va);
                    chunk(vb, c + 1);
                }
                flag = !(m1 >= sk.G1) || !(m2 >= sk.G2) || !(qn > 0.0f);
            } else {
                const float sa = pa * __frcp_rn(den);
                float m = __int_as_float(0x7f800000);
                // words 4c .. 4c + 3, eight coordinates each: pairs of even
                // coordinates collect in b0, of odd ones in b1
                auto chunk = [&](const uint32_t (&v)[32], int c) {
                    uint32_t o1[4], o2[4];
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        uint32_t b0 = 0u, b1 = 0u;
#pragma unroll
                        for (int e = 0; e < 8; e += 2) {
                            b0 = __funnelshift_r(b0, pair_code_s(__uint_as_float(v[8 * w + e]), sa, pbc, den, tab, m), 8);
                            b1 = __funnelshift_r(b1, pair_code_s(__uint_as_float(v[8 * w + e + 1]), sa, pbc, den, tab, m), 8);
                        }
                        o1[w] = (b0 & 0x0F0F0F0Fu) | ((b1 & 0x0F0F0F0Fu) << 4);
                        o2[w] = ((b0 >> 4) & 0x0F0F0F0Fu) | (b1 & 0xF0F0F0F0u);
                    }
                    if (okrow) {
                        *reinterpret_cast<uint4 *>(d1 + 4 * c) = make_uint4(o1[0], o1[1], o1[2], o1[3]);
                        *reinterpret_cast<uint4 *>(d2 + 4 * c) = make_uint4(o2[0], o2[1], o2[2], o2[3]);
                    }
                };
                qt_ld32(tl, va);
#pragma unroll 1
                for (int c = 0; c < 4; c += 2) {
                    qt_wait_ld();
                    qt_hold(va);
                    qt_ld32(tl + 32 * (c + 1), vb);
                    chunk(va, c);
                    qt_wait_ld();
                    qt_hold(vb);
                    if (c + 2 < 4) qt_ld32(tl + 32 * (c + 2), va);
                    chunk(vb, c + 1);
                }
                flag = !(m >= p.guard * den) || !(qn > 0.0f);
            }
            // the accumulator buffer is free for tile i + TE_G
            qt_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[g]);

            flag = flag && okrow;
            if (okrow && !flag) p.norms[drow] = n;
            // rows inside the guard band go to the list (this thread's fast
            // words ordered before their exact ones by the fence and the list
            // entry) while it has room; else the warp recomputes them here.
            // The b = 4 books flag ~2 % of rows, more than the two fixup
            // warps keep up with: the rest wait for the epilogue warps, which
            // drain the list with them once their tiles are done (measured:
            // better than recomputing the excess in the epilogue at once,
            // which held the MMA pipeline)
            bool here = false;
            if (flag) {
                // the recompute reads the row again: start bringing it to L1
                const char *xr = static_cast<const char *>(p.x) + (size_t)row * ROW_BYTES;
                asm volatile("prefetch.global.L1 [%0];" ::"l"(xr));
                asm volatile("prefetch.global.L1 [%0];" ::"l"(xr + 128));
                __threadfence_block();
                const uint32_t k = atomicAdd(fq_n, 1u);
                if (k < (uint32_t)TE_FQ)
                    fq[k] = (uint32_t)row + 1u;
                else
                    here = true;
            }
            __syncwarp();  // the fast words of a flagged row are written before its exact ones
            unsigned fl = __ballot_sync(FULL_MASK, here);
            while (fl) {
                const int bit = __ffs(fl) - 1;
                fl &= fl - 1;
                fixup_one<MODE>(p, t * TE_M + 32 * q + bit, lane, fb);
            }
            __syncwarp();
        }
        __syncwarp();
        if (lane == 0) {
            __threadfence_block();
            atomicAdd(fq_done, 1u);
        }
        drain(fb);
    } else {
        // ---- fixup warps
        drain(fix_books<MODE>(p, lane));
    }

    qt_fence_before();
    __syncthreads();
    qt_fence_after();
    if (warp == 1) tmem_free(tmem, 512);
}

}  // namespace
}  // namespace vq
