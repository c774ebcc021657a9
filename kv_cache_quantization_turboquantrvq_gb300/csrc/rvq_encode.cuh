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
// The library's books have encoders of their own, with the same rings and
// exact recompute, the rotation on the tensor cores and four lanes per row:
// rvq_encode_sym2_kernel for symmetric 4-level books (b = 2) and
// rvq_encode_pair4_kernel for 16-level books with a pair table (b = 4).
//
// The including translation unit defines VQ_RVQ_ERR, the device error word
// the bodies report into (VQ_DEVERR_* bits).
#pragma once

#include <cuda_fp16.h>

#include "device_common.cuh"
#include "launch.h"

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
    static_assert(!(MODE == MODE_SYM && BITS == 2), "symmetric b = 2 books: rvq_encode_sym2_kernel");
    static_assert(MODE != MODE_PAIR, "the b = 4 pair table: rvq_encode_pair4_kernel");
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

// ------------------------------------------- encode, symmetric b = 2, tensor cores
//
// The same pass as rvq_encode_kernel for symmetric 4-level books, with the
// rotation on the tensor cores.  Write a coordinate as c = 8a + b (a < 16,
// b < 8); the Sylvester matrix factors as H128[8a' + b'][8a + b] =
// H16[a'][a] H8[b'][b].  Per warp and 16-row block, for each b the product
// T_b = X_b H16 (X_b: the 16 rows' values x[8a + b], a as the k index) is one
// pair of 16x8x16 mma.sync (fp16 operands, exact +-1 products, fp32
// accumulation); then the H8 factor is three fp32x2 butterfly stages across
// the eight accumulator tiles, in registers.  The columns of the H16 operand
// are permuted so that the lane with t4 = lane & 3 receives a' = 4 t4 ..
// 4 t4 + 3, i.e. output coordinates 32 t4 .. 32 t4 + 31: two whole code words
// of each of its two rows (g8 = lane >> 2 and g8 + 8), so no word is split
// across lanes.  The A operands come from 16-byte reads of the swizzled
// staged rows (chunk a of row r holds x[8a .. 8a + 7]) and one byte permute
// per register.  The norm is taken from the H16 outputs (their squares sum to
// 16 sum x^2), the quantizer is sym2_code2, rows with a value in the guard
// band go to rvq_fixup_row.
constexpr int S2_WARPS = 16;
constexpr int S2_STAGES = 3;

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// fp16 pair (+-1 of H16[a][a'], H16[a + 1][a']) for the B operand
__device__ __forceinline__ uint32_t h16_pair(int a, int ap)
{
    const uint32_t lo = (__popc(a & ap) & 1) ? 0xBC00u : 0x3C00u;
    const uint32_t hi = (__popc((a + 1) & ap) & 1) ? 0xBC00u : 0x3C00u;
    return lo | (hi << 16);
}

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

// S = X H128 for rows g8 and g8 + 8 of a staged 16-row block: the A operands
// from 16-byte reads of the swizzled rows (chunk a of a row holds
// x[8a .. 8a + 7]) and one byte permute per register, X_b H16 for b = 0..7 as
// 16x8x16 mma.sync with the permuted H16 columns in hb, the rows' sums of
// squares (q0, q1) from the H16 outputs, then H8 as three butterfly stages
// across b.  Afterwards acc[b'][nt][2r + e] = S at coordinate
// 32 t4 + 16 nt + 8 e + b' of row g8 + 8r.
template <bool SGN>
__device__ __forceinline__ void tc_rotate_block(const unsigned char *sbuf, const uint4 *ssg, const uint32_t (&hb)[2][2],
                                                int g8, int t4, float (&acc)[8][2][4], float &q0, float &q1)
{
    // ---- T_b = X_b H16 for b = 0..7 on the tensor cores
    {
        // u[r][j]: row g8 + 8r, chunk a = 2 t4 + {0, 1, 8, 9}[j]
        uint4 u[2][4];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int a = 2 * t4 + (j & 1) + 8 * (j >> 1);
                u[r][j] = *reinterpret_cast<const uint4 *>(sbuf + (j >> 1) * (ENC_BLOCK / 2) + swz128(g8 + 8 * r, a & 7));
                if constexpr (SGN) {
                    const uint4 m = ssg[a];
                    u[r][j] = make_uint4(u[r][j].x ^ m.x, u[r][j].y ^ m.y, u[r][j].z ^ m.z, u[r][j].w ^ m.w);
                }
            }
        }
#pragma unroll
        for (int b = 0; b < 8; ++b) {
            const uint32_t sel = (b & 1) ? 0x7632u : 0x5410u;
            auto word = [&](const uint4 &v) -> uint32_t {
                return (b >> 1) == 0 ? v.x : (b >> 1) == 1 ? v.y : (b >> 1) == 2 ? v.z : v.w;
            };
            const uint32_t a0 = __byte_perm(word(u[0][0]), word(u[0][1]), sel);
            const uint32_t a1 = __byte_perm(word(u[1][0]), word(u[1][1]), sel);
            const uint32_t a2 = __byte_perm(word(u[0][2]), word(u[0][3]), sel);
            const uint32_t a3 = __byte_perm(word(u[1][2]), word(u[1][3]), sel);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                acc[b][nt][0] = acc[b][nt][1] = acc[b][nt][2] = acc[b][nt][3] = 0.0f;
                mma_f16_16816(acc[b][nt], a0, a1, a2, a3, hb[nt][0], hb[nt][1]);
            }
        }
    }

    // ---- norms: the H16 outputs' squares sum to 16 sum x^2 (per row)
    {
        float2 s0 = make_float2(0.0f, 0.0f), s1 = s0;
#pragma unroll
        for (int b = 0; b < 8; ++b) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const float2 v0 = make_float2(acc[b][nt][0], acc[b][nt][1]);
                const float2 v1 = make_float2(acc[b][nt][2], acc[b][nt][3]);
                s0 = __ffma2_rn(v0, v0, s0);
                s1 = __ffma2_rn(v1, v1, s1);
            }
        }
        q0 = s0.x + s0.y;
        q1 = s1.x + s1.y;
        q0 += __shfl_xor_sync(FULL_MASK, q0, 1);
        q1 += __shfl_xor_sync(FULL_MASK, q1, 1);
        q0 += __shfl_xor_sync(FULL_MASK, q0, 2);
        q1 += __shfl_xor_sync(FULL_MASK, q1, 2);
        q0 *= 0.0625f;
        q1 *= 0.0625f;
    }
    // ---- H8 across b: acc[b'][nt] = S at coordinates 32 t4 + 16 nt + b' (.x / c2)
    // and 32 t4 + 16 nt + 8 + b' (.y / c3)
    const float2 neg1 = make_float2(-1.0f, -1.0f);
#pragma unroll
    for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
        for (int b = 0; b < 8; ++b) {
            if ((b & h) == 0) {
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        const float2 x = make_float2(acc[b][nt][2 * r], acc[b][nt][2 * r + 1]);
                        const float2 y = make_float2(acc[b + h][nt][2 * r], acc[b + h][nt][2 * r + 1]);
                        const float2 sum = __fadd2_rn(x, y);
                        const float2 dif = __ffma2_rn(y, neg1, x);
                        acc[b][nt][2 * r] = sum.x;
                        acc[b][nt][2 * r + 1] = sum.y;
                        acc[b + h][nt][2 * r] = dif.x;
                        acc[b + h][nt][2 * r + 1] = dif.y;
                    }
                }
            }
        }
    }
}

template <bool SGN>
__device__ __forceinline__ void rvq_encode_sym2_body(const RvqEncodeParams &p, int cta, int ncta)
{
    constexpr int W = D * 2 / 32;  // 8 words per row and stream
    extern __shared__ __align__(128) unsigned char smem_raw[];
    unsigned char *base = smem_1k(smem_raw);
    uint4 *ssg = reinterpret_cast<uint4 *>(base);  // sign masks: chunk a = coordinates 8a .. 8a + 7
    unsigned char *smem = base + ENC_SGN_BYTES;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g8 = lane >> 2, t4 = lane & 3;
    unsigned char *ring = smem + warp * (S2_STAGES * ENC_BLOCK);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + S2_WARPS * S2_STAGES * ENC_BLOCK) + warp * S2_STAGES;

    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < S2_STAGES; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    if (threadIdx.x < 16) {
        const int c0 = 8 * threadIdx.x;
        ssg[threadIdx.x] = make_uint4(half2_sign_mask(sign_pair(p.sgn, c0)), half2_sign_mask(sign_pair(p.sgn, c0 + 2)),
                                      half2_sign_mask(sign_pair(p.sgn, c0 + 4)), half2_sign_mask(sign_pair(p.sgn, c0 + 6)));
    }
    __syncthreads();

    const uint64_t pol = l2_policy_evict_first();
    // shuffle tables of the exact recompute
    const float tb1 = p.t1.bnd[lane];
    const int tc1 = p.t1.code[lane];
    const float tb2 = p.t2.bnd[lane];
    const int tc2 = p.t2.code[lane];
    const float tcen = p.c1[lane & 3];
    // unit-norm book constants: B, E, B - c2, c3 - c2, 2 / B, 2 / E
    const float b1u = p.b1[2], b2u = p.b2[2];
    const float bc2u = p.b1[2] - p.c1[2], dcu = p.c1[3] - p.c1[2];
    const float kb1 = __fdiv_rn(2.0f, b1u), kb2 = __fdiv_rn(2.0f, b2u);
    // B operand: column n = g8 of n-tile nt is a' = 4 (g8 >> 1) + 2 nt + (g8 & 1);
    // b0 holds k = 2 t4, 2 t4 + 1 and b1 k = 2 t4 + 8, 2 t4 + 9
    uint32_t hb[2][2];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        const int ap = 4 * (g8 >> 1) + 2 * nt + (g8 & 1);
        hb[nt][0] = h16_pair(2 * t4, ap);
        hb[nt][1] = h16_pair(2 * t4 + 8, ap);
    }

    const int nblk = (p.N + ER - 1) / ER;
    const int gw = cta * S2_WARPS + warp;
    const int tw = ncta * S2_WARPS;
    // destination row = source row (no batch offsets, same capacity)
    const bool dense = p.dst_off == nullptr && p.S_dst == p.S && p.S_q == p.S;
    auto issue = [&](int blk, int s) {
        if (lane == 0) {
            mbar_arrive_expect_tx(&bars[s], (uint32_t)ENC_BLOCK);
            tma_load_2d(ring + s * ENC_BLOCK, &p.tmap, 0, blk * ER, &bars[s], pol);
            tma_load_2d(ring + s * ENC_BLOCK + ENC_BLOCK / 2, &p.tmap, 64, blk * ER, &bars[s], pol);
        }
    };
#pragma unroll
    for (int s = 0; s < S2_STAGES; ++s) {
        const int blk = gw + s * tw;
        if (blk < nblk) issue(blk, s);
    }

    int s = 0;
    uint32_t ph = 0;
    for (int it = 0;; ++it) {
        const int blk = gw + it * tw;
        if (blk >= nblk) break;
        const bool ok = mbar_wait_bounded(&bars[s], ph);
        if (!__all_sync(FULL_MASK, ok)) {
            if (lane == 0) atomicOr(&VQ_RVQ_ERR, (unsigned)VQ_DEVERR_WAIT_TIMEOUT);
            for (int k = 1; k < S2_STAGES; ++k) {
                const int it2 = it + k;
                if (gw + it2 * tw < nblk)
                    (void)mbar_wait_bounded(&bars[it2 % S2_STAGES], (uint32_t)(it2 / S2_STAGES) & 1u);
            }
            return;
        }
        const unsigned char *sbuf = ring + s * ENC_BLOCK;

        float acc[8][2][4];
        float q0, q1;
        tc_rotate_block<SGN>(sbuf, ssg, hb, g8, t4, acc, q0, q1);
        const float n0 = __fsqrt_rn(q0), n1 = __fsqrt_rn(q1);
        const float den0 = n0 * SQRT_D_HI, den1 = n1 * SQRT_D_HI;

        // ---- quantize: word 2 t4 + nt of row g8 + 8r gets b' = 0..7 of .x at
        // positions 0..7 and of .y at positions 8..15
        const SymRow sk0 = sym2_row(den0, p.guard * den0, b1u, b2u, bc2u, dcu, kb1, kb2);
        const SymRow sk1 = sym2_row(den1, p.guard * den1, b1u, b2u, bc2u, dcu, kb1, kb2);
        // running minima of the stage-1 / stage-2 margin products of each row
        float m0a = __int_as_float(0x7f800000), m0b = m0a, m1a = m0a, m1b = m0a;
        uint32_t w1[2][2], w2[2][2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                uint32_t a1x = 0u, a2x = 0u, a1y = 0u, a2y = 0u;
#pragma unroll
                for (int b = 7; b >= 0; --b) {
                    const float2 y2 = make_float2(acc[b][nt][2 * r], acc[b][nt][2 * r + 1]);
                    if (r == 0) sym2_code2(y2, sk0, a1x, a2x, a1y, a2y, m0a, m0b);
                    else sym2_code2(y2, sk1, a1x, a2x, a1y, a2y, m1a, m1b);
                }
                sym2_words(__byte_perm(a1x, a1y, 0x5410u), __byte_perm(a2x, a2y, 0x5410u), w1[r][nt], w2[r][nt]);
            }
        }

        // ---- guard band: a row is flagged if any of its four lanes saw a value
        // inside the band (and always when it is zero)
        const int row0 = blk * ER + g8, row1 = row0 + 8;
        const bool valid0 = row0 < p.N, valid1 = row1 < p.N;
        const bool f0 = valid0 && (!(m0a >= sk0.G1) || !(m0b >= sk0.G2) || !(q0 > 0.0f));
        const bool f1 = valid1 && (!(m1a >= sk1.G1) || !(m1b >= sk1.G2) || !(q1 > 0.0f));
        int f = (f0 ? 1 : 0) | (f1 ? 2 : 0);
        f |= __shfl_xor_sync(FULL_MASK, f, 1);
        f |= __shfl_xor_sync(FULL_MASK, f, 2);

        // ---- fast words: 8 bytes per lane, row and stream (a block's 16 rows are
        // contiguous in both streams)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int row = r ? row1 : row0;
            size_t drow = (size_t)row;
            if ((r ? valid1 : valid0) && !(f & (1 << r)) && (dense || rvq_dst_row(p, row, drow))) {
                *reinterpret_cast<uint2 *>(p.p1 + drow * W + 2 * t4) = make_uint2(w1[r][0], w1[r][1]);
                *reinterpret_cast<uint2 *>(p.p2 + drow * W + 2 * t4) = make_uint2(w2[r][0], w2[r][1]);
                if (t4 == 0) p.norms[drow] = r ? n1 : n0;
            }
        }

        // ---- flagged rows: exact recompute by the warp
        unsigned fl = (__ballot_sync(FULL_MASK, (f & 1) != 0) & 0x11111111u) |
                      ((__ballot_sync(FULL_MASK, (f & 2) != 0) & 0x11111111u) << 1);
        while (fl) {
            const int bit = __ffs(fl) - 1;
            fl &= fl - 1;
            const int r = (bit >> 2) + 8 * (bit & 1);
            rvq_fixup_row<2, false>(p, sbuf, r, blk * ER + r, lane, tb1, tc1, tb2, tc2, tcen);
        }
        __syncwarp();

        fence_proxy_async_smem();
        {
            const int nb = blk + S2_STAGES * tw;
            if (nb < nblk) issue(nb, s);
        }
        if (++s == S2_STAGES) {
            s = 0;
            ph ^= 1u;
        }
    }
}

// ------------------------------------------- encode, b = 4 pair table, tensor cores
//
// The rotation of rvq_encode_sym2_kernel (tc_rotate_block) with the
// 16-level quantizer of the pair table (PairTable in launch.h): one cell
// lookup per coordinate gives both codes.  The table lives in shared memory
// replicated P4_REP = 16 times (cell g, replica j at byte (16 g + j) 8) and
// lane l reads replica l & 15: an 8-byte read is served per half-warp, so the
// 16 lanes of each half always hit 16 distinct bank pairs and the lookup is
// free of bank conflicts.  The quantizer works on S = H x directly: with
// den = n sqrt(D), y > bnd exactly when bnd den - S is negative (one FMA
// rounding of an exact product-difference), the cell coordinate is
// fma(S, a / den, bc), and the margin |bnd den - S| is compared with
// guard den; the host builds the table with every step at least three guard
// bands inside its cell, which absorbs the rounding of a / den (the cell a
// value lands in can differ from the y-domain map only near cell edges,
// where the neighbouring cell's entry gives the same pair).  After the
// rotation acc[b'][nt][2r + e], b' = 0..7, are the eight coordinates of word
// 4 t4 + 2 nt + e of row g8 + 8r, so each lane packs and stores four whole
// words per row and stream.  Rows with a value inside the guard band go to
// rvq_fixup_row.
constexpr int P4_STAGES = 2;
constexpr int P4_REP = 16;
constexpr int P4_TAB_BYTES = PT_CELLS * P4_REP * 8;

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

template <bool SGN>
__device__ __forceinline__ void rvq_encode_pair4_body(const RvqEncodeParams &p, int cta, int ncta)
{
    constexpr int W = D * 4 / 32;  // 16 words per row and stream
    extern __shared__ __align__(128) unsigned char smem_raw[];
    unsigned char *base = smem_1k(smem_raw);
    uint4 *ssg = reinterpret_cast<uint4 *>(base);  // sign masks: chunk a = coordinates 8a .. 8a + 7
    uint2 *ptab = reinterpret_cast<uint2 *>(base + ENC_SGN_BYTES);
    unsigned char *smem = base + ENC_SGN_BYTES + P4_TAB_BYTES;  // 1024-byte aligned
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g8 = lane >> 2, t4 = lane & 3;
    unsigned char *ring = smem + warp * (P4_STAGES * ENC_BLOCK);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + S2_WARPS * P4_STAGES * ENC_BLOCK) + warp * P4_STAGES;

    const uint64_t pol = l2_policy_evict_first();
    const int nblk = (p.N + ER - 1) / ER;
    const int gw = cta * S2_WARPS + warp;
    const int tw = ncta * S2_WARPS;
    auto issue = [&](int blk, int s) {
        if (lane == 0) {
            mbar_arrive_expect_tx(&bars[s], (uint32_t)ENC_BLOCK);
            tma_load_2d(ring + s * ENC_BLOCK, &p.tmap, 0, blk * ER, &bars[s], pol);
            tma_load_2d(ring + s * ENC_BLOCK + ENC_BLOCK / 2, &p.tmap, 64, blk * ER, &bars[s], pol);
        }
    };
    // the warp's barriers, then its first blocks in flight while the CTA
    // fills the sign masks and the replicated table
    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < P4_STAGES; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
#pragma unroll
        for (int s = 0; s < P4_STAGES; ++s) {
            const int blk = gw + s * tw;
            if (blk < nblk) issue(blk, s);
        }
    }
    if (threadIdx.x < 16) {
        const int c0 = 8 * threadIdx.x;
        ssg[threadIdx.x] = make_uint4(half2_sign_mask(sign_pair(p.sgn, c0)), half2_sign_mask(sign_pair(p.sgn, c0 + 2)),
                                      half2_sign_mask(sign_pair(p.sgn, c0 + 4)), half2_sign_mask(sign_pair(p.sgn, c0 + 6)));
    }
    for (int i = threadIdx.x; i < PT_CELLS * P4_REP; i += blockDim.x) ptab[i] = p.pt.ent[i / P4_REP];
    __syncthreads();

    // shuffle tables of the exact recompute
    const float tb1 = p.t1.bnd[lane];
    const int tc1 = p.t1.code[lane];
    const float tb2 = p.t2.bnd[lane];
    const int tc2 = p.t2.code[lane];
    const float tcen = p.c1[lane & 15];
    const float pa = p.pt.a, pbc = p.pt.bc;
    const uint32_t tab = smem_u32(ptab) + 8u * (uint32_t)(lane & (P4_REP - 1)) - (0x4B400000u << 7);
    uint32_t hb[2][2];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        const int ap = 4 * (g8 >> 1) + 2 * nt + (g8 & 1);
        hb[nt][0] = h16_pair(2 * t4, ap);
        hb[nt][1] = h16_pair(2 * t4 + 8, ap);
    }

    // destination row = source row (no batch offsets, same capacity)
    const bool dense = p.dst_off == nullptr && p.S_dst == p.S && p.S_q == p.S;

    int s = 0;
    uint32_t ph = 0;
    for (int it = 0;; ++it) {
        const int blk = gw + it * tw;
        if (blk >= nblk) break;
        const bool ok = mbar_wait_bounded(&bars[s], ph);
        if (!__all_sync(FULL_MASK, ok)) {
            if (lane == 0) atomicOr(&VQ_RVQ_ERR, (unsigned)VQ_DEVERR_WAIT_TIMEOUT);
            for (int k = 1; k < P4_STAGES; ++k) {
                const int it2 = it + k;
                if (gw + it2 * tw < nblk)
                    (void)mbar_wait_bounded(&bars[it2 % P4_STAGES], (uint32_t)(it2 / P4_STAGES) & 1u);
            }
            return;
        }
        const unsigned char *sbuf = ring + s * ENC_BLOCK;

        float acc[8][2][4];
        float q0, q1;
        tc_rotate_block<SGN>(sbuf, ssg, hb, g8, t4, acc, q0, q1);
        const float n0 = __fsqrt_rn(q0), n1 = __fsqrt_rn(q1);
        // per row: den = n sqrt(D), the cell slope a / den and the margin
        // threshold guard den (a zero row gives den = 0 and is always flagged)
        const float den0 = n0 * SQRT_D_HI, den1 = n1 * SQRT_D_HI;
        const float sa0 = pa * __frcp_rn(den0), sa1 = pa * __frcp_rn(den1);

        // ---- quantize: word 2 nt + e of the lane (word 4 t4 + 2 nt + e of the
        // row) from b' = 0..7 of acc[.][nt][2r + e]; the pairs i1 | i2 << 4 of
        // even coordinates collect in b0, of odd ones in b1 (first at byte 0),
        // then the low nibbles make the stage-1 word and the high nibbles the
        // stage-2 word
        float m0 = __int_as_float(0x7f800000), m1 = m0;
        uint32_t w1[2][4], w2[2][4];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const float sa = r ? sa1 : sa0, den = r ? den1 : den0;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                uint32_t b0[2] = {0u, 0u}, b1[2] = {0u, 0u};
#pragma unroll
                for (int b = 0; b < 8; ++b) {
                    const uint32_t px = pair_code_s(acc[b][nt][2 * r], sa, pbc, den, tab, r ? m1 : m0);
                    const uint32_t py = pair_code_s(acc[b][nt][2 * r + 1], sa, pbc, den, tab, r ? m1 : m0);
                    if (b & 1) {
                        b1[0] = __funnelshift_r(b1[0], px, 8);
                        b1[1] = __funnelshift_r(b1[1], py, 8);
                    } else {
                        b0[0] = __funnelshift_r(b0[0], px, 8);
                        b0[1] = __funnelshift_r(b0[1], py, 8);
                    }
                }
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    w1[r][2 * nt + e] = (b0[e] & 0x0F0F0F0Fu) | ((b1[e] & 0x0F0F0F0Fu) << 4);
                    w2[r][2 * nt + e] = ((b0[e] >> 4) & 0x0F0F0F0Fu) | (b1[e] & 0xF0F0F0F0u);
                }
            }
        }

        // ---- guard band: a row is flagged if any of its four lanes saw a value
        // inside the band (and always when it is zero)
        const int row0 = blk * ER + g8, row1 = row0 + 8;
        const bool valid0 = row0 < p.N, valid1 = row1 < p.N;
        const bool f0 = valid0 && (!(m0 >= p.guard * den0) || !(q0 > 0.0f));
        const bool f1 = valid1 && (!(m1 >= p.guard * den1) || !(q1 > 0.0f));
        int f = (f0 ? 1 : 0) | (f1 ? 2 : 0);
        f |= __shfl_xor_sync(FULL_MASK, f, 1);
        f |= __shfl_xor_sync(FULL_MASK, f, 2);

        // ---- fast words: 16 bytes per lane, row and stream (a block's 16 rows
        // are contiguous in both streams)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int row = r ? row1 : row0;
            size_t drow = (size_t)row;
            if ((r ? valid1 : valid0) && !(f & (1 << r)) && (dense || rvq_dst_row(p, row, drow))) {
                *reinterpret_cast<uint4 *>(p.p1 + drow * W + 4 * t4) = make_uint4(w1[r][0], w1[r][1], w1[r][2], w1[r][3]);
                *reinterpret_cast<uint4 *>(p.p2 + drow * W + 4 * t4) = make_uint4(w2[r][0], w2[r][1], w2[r][2], w2[r][3]);
                if (t4 == 0) p.norms[drow] = r ? n1 : n0;
            }
        }

        // ---- flagged rows: exact recompute by the warp
        unsigned fl = (__ballot_sync(FULL_MASK, (f & 1) != 0) & 0x11111111u) |
                      ((__ballot_sync(FULL_MASK, (f & 2) != 0) & 0x11111111u) << 1);
        while (fl) {
            const int bit = __ffs(fl) - 1;
            fl &= fl - 1;
            const int r = (bit >> 2) + 8 * (bit & 1);
            rvq_fixup_row<4, true>(p, sbuf, r, blk * ER + r, lane, tb1, tc1, tb2, tc2, tcen);
        }
        __syncwarp();

        fence_proxy_async_smem();
        {
            const int nb = blk + P4_STAGES * tw;
            if (nb < nblk) issue(nb, s);
        }
        if (++s == P4_STAGES) {
            s = 0;
            ph ^= 1u;
        }
    }
}

}  // namespace
}  // namespace vq
