// kivi_quant.cuh - KIVI quantize+pack device code for sm_103a, shared by the
// quantize kernels (kivi.cu) and the fused decode-time flush (flush.cu).
// Each body runs one CTA's share of a persistent grid (CTA `cta` of `ncta`,
// WARPS warps per CTA).
//
// Method (VeloxQuant-MLX blog, tag "kivi", first post "What we're actually
// optimizing" and second post "What KIVI is"): per group zero = min,
// scale = (max - min)/(2^b - 1), q = round((x - zero)/scale) with ties to even
// ("Rounding mode"), recon = q*scale + zero.  Keys: groups of G tokens per
// channel; values: groups of G channels per token; only tokens [0, S_q) are
// flushed, the residual window [S_q, S) stays fp16 and is not touched.
//
// The pages quantize and immediately dequantize to fp16; here the codes are
// packed (LSB first, 32/b per uint32) with fp16 scale and zero per group, the
// storage step the pages name as the next one.
//
// Exactness: codes are those of the exact quotient
//   t = (x - min)(2^b - 1)/(max - min), rounded half to even.
// With A = x - min, R = max - min and C = 2^b - 1, the code is decided against
// the two half-integers around the fp32 estimate r = rint(A * C/R) by the
// signs of C*A - (r -+ 1/2)*R, each formed by one FMA.  When R is exact in
// fp32 with at most 19 significant bits, every exact tie has A and C*A exact in
// fp32, so those signs (and zeros) are exact; other groups are decided in
// 64-bit integers.  No per-element branch and no binary64 on the common path.
// The stored scale is fp16(fp32(range/(2^b - 1))) with both roundings to
// nearest even.
//
// Values (per token): two threads per row (64 channels each), 16-row blocks
// staged as two swizzled TMA boxes into a per-warp ring (as the RVQ encoder).
// Keys (per channel): one [G x 64] half-tile per warp step as one TMA box; lane
// l owns two channels and walks the G tokens, so no cross-thread reduction is
// needed (the pages' "one thread, one whole group").
//
// Dequant: one fp16x2 fused multiply-add per element pair, q * scale + zero
// rounded once from its exact value (fma.rn.f16x2), the code entering exactly
// as (1024 + q) - 1024 in fp16.
//
// The including translation unit defines VQ_KIVI_ERR, the device error word
// the bodies report into (VQ_DEVERR_* bits).
#pragma once

#include <cuda_fp16.h>

#include "device_common.cuh"
#include "launch.h"

#ifndef VQ_KIVI_ERR
#error "define VQ_KIVI_ERR (the device error word) before including kivi_quant.cuh"
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
constexpr float MAGIC = 12582912.0f;  // 1.5 * 2^23: x + MAGIC rounds x to an integer, ties to even

// ------------------------------------------------------------ group scalars

struct GroupQ {
    float mn;      // group minimum (exact)
    float f;       // (2^b - 1) / (max - min) in fp32, 0 for a constant group
    float rr;      // max - min in fp32
    bool fast;     // rr exact with <= 19 significant bits: the FMA test is exact
    __half scale_h, zero_h;
};

// 1.5 * 2^23 - 1: fma(A, f, MAGIC1) holds MAGIC - 1 + rint(A f) exactly.
constexpr float MAGIC1 = 12582911.0f;
// Saturated step: sat(z * 2^40 + 1/2) is 0 for z < 0, 1/2 for z == 0 and 1 for
// z > 0 whenever |z| >= 2^-41; the tie quantities below are multiples of
// 2^-25 (fp16 data), so nothing smaller than that occurs.
constexpr float STEP_SCALE = 1099511627776.0f;

__device__ __forceinline__ float step_half(float z)
{
    return __saturatef(fmaf(z, STEP_SCALE, 0.5f));
}

// RN32 of the exact (mx - mn)/c, given fp16-valued mx > mn.
__device__ __noinline__ float exact_scale32_slow(float mx, float mn, float c)
{
    const double d = (double)mx - (double)mn;  // exact: fp16 values
    const double q = d / (double)c;
    float f = (float)q;
    const float up = __int_as_float(__float_as_int(f) + 1);
    const float dn = __int_as_float(__float_as_int(f) - 1);
    const float other = (double)f > q ? dn : up;
    const double mid = 0.5 * ((double)f + (double)other);
    if (q == mid) {
        const double rem = fma(-q, (double)c, d);
        if (rem > 0.0) return (double)f > (double)other ? f : other;
        if (rem < 0.0) return (double)f < (double)other ? f : other;
    }
    return f;
}

template <int BITS>
__device__ __forceinline__ GroupQ group_setup(float mn, float mx)
{
    constexpr float C = (float)((1 << BITS) - 1);
    GroupQ g;
    g.mn = mn;
    g.zero_h = __float2half_rn(mn);  // exact: mn is an fp16 value
    if (mx > mn) {
        float d, e;
        two_sum(mx, -mn, d, e);
        g.rr = d;
        g.fast = e == 0.0f && (__float_as_uint(d) & 31u) == 0u;
        const float s32 = (e == 0.0f) ? __fdiv_rn(d, C) : exact_scale32_slow(mx, mn, C);
        g.scale_h = __float2half_rn(s32);
        g.f = __fdiv_rn(C, d);
    } else {
        g.rr = 0.0f;
        g.fast = true;
        g.scale_h = __float2half_rn(0.0f);
        g.f = 0.0f;
    }
    return g;
}

// Code of t = (x - mn) C / R, ties to even, in 64-bit integers: fp16 values
// times 2^24 are integers below 2^40, so 2 C A - (2j + 1) R is exact.
template <int BITS>
__device__ __noinline__ uint32_t code_int64(float x, float mn, float mx)
{
    const long long C = (1 << BITS) - 1;
    const long long X = __float2ll_rn(x * 16777216.0f);
    const long long MN = __float2ll_rn(mn * 16777216.0f);
    const long long R = __float2ll_rn(mx * 16777216.0f) - MN;
    if (R == 0) return 0u;
    const long long A = X - MN;
    uint32_t q = 0;
    for (int j = 0; j < (int)C; ++j) {
        const long long Z = 2 * C * A - (2LL * j + 1) * R;
        q += (Z > 0 || (Z == 0 && (j & 1))) ? 1u : 0u;
    }
    return q;
}

// Exact codes of two elements of a `fast` group, returned in the low bits of
// qa / qb.  With r = rint(A f) (the fp32 estimate of t rounded), u = C A - r R,
//   q = r - 1 + step(u + R/2) + step(u - R/2)
// where step is 0 / 1/2 / 1 for a negative / zero / positive argument: the two
// terms test t against r - 1/2 and r + 1/2 (exact signs when C A and R are
// exact, which holds for every exact tie of a fast group), and a tie leaves a
// half that the final round-to-nearest-even addition resolves to the even
// neighbour.  Everything runs on the FMA pipe, two elements per instruction
// where the operation exists for fp32 pairs.
template <int BITS>
__device__ __forceinline__ void code_pair2(__half a, __half b, float2 mn, float2 f, float2 rr, uint32_t &qa,
                                           uint32_t &qb)
{
    constexpr float C = (float)((1 << BITS) - 1);
    const float2 A = make_float2(add_f16_f32(a, -mn.x), add_f16_f32(b, -mn.y));
    const float2 tm = __ffma2_rn(A, f, make_float2(MAGIC1, MAGIC1));
    const float2 r = __fadd2_rn(tm, make_float2(-MAGIC1, -MAGIC1));
    const float2 ca = __fmul2_rn(A, make_float2(C, C));
    const float2 u = __ffma2_rn(r, make_float2(-rr.x, -rr.y), ca);
    const float2 h = make_float2(0.5f * rr.x, 0.5f * rr.y);
    const float2 zl = __fadd2_rn(u, h);
    const float2 zr = __fadd2_rn(u, make_float2(-h.x, -h.y));
    const float2 st = __fadd2_rn(make_float2(step_half(zl.x), step_half(zl.y)),
                                 make_float2(step_half(zr.x), step_half(zr.y)));
    const float2 qm = __fadd2_rn(tm, st);  // MAGIC + q, ties to even
    qa = __float_as_uint(qm.x);
    qb = __float_as_uint(qm.y);
}

template <int BITS>
__device__ __forceinline__ void code_pair(__half a, __half b, const GroupQ &g, uint32_t &qa, uint32_t &qb)
{
    code_pair2<BITS>(a, b, make_float2(g.mn, g.mn), make_float2(g.f, g.f), make_float2(g.rr, g.rr), qa, qb);
}

// ------------------------------------------------------------ fast codes
//
// The common path takes q = rint(A f) with A = fl(x - min) and
// f = fl((2^b - 1)/fl(max - min)).  A f differs from the exact t by three
// relative roundings, at most 3 * 2^-24 * t < 2^-18.4 for t <= 15, so when
// |rint(A f) - A f| < 1/2 - 2^-16 the estimate rounds like t.  The test is
// e = rint(A f) - A f (one FMA, one rounding) and the sign of e^2 - THR with
// THR = (1/2 - 2^-16)^2; the sign bits of all elements of a word are ANDed,
// so a clear sign bit sends the word to the exact path (code_pair /
// code_int64 above).  Random data trips it for about 3e-5 of the elements;
// exact ties always trip it.
constexpr float TIE_THR = (float)((0.5 - 1.0 / 65536.0) * (0.5 - 1.0 / 65536.0));

// Codes of two elements (MAGIC-biased: the low bits of qa / qb are the codes)
// and the running AND of the tie-test sign bits.
__device__ __forceinline__ void code_pair_fast(__half a, __half b, float mna, float mnb, float2 f,
                                               float2 nf, uint32_t &qa, uint32_t &qb, uint32_t &ok)
{
    const float2 A = make_float2(add_f16_f32(a, -mna), add_f16_f32(b, -mnb));
    const float2 tm = __ffma2_rn(A, f, make_float2(MAGIC, MAGIC));
    const float2 r = __fadd2_rn(tm, make_float2(-MAGIC, -MAGIC));
    const float2 e = __ffma2_rn(A, nf, r);
    const float2 c = __ffma2_rn(e, e, make_float2(-TIE_THR, -TIE_THR));
    ok &= __float_as_uint(c.x) & __float_as_uint(c.y);
    qa = __float_as_uint(tm.x);
    qb = __float_as_uint(tm.y);
}

// Exact code of one element (the slow path of a word).
template <int BITS>
__device__ __noinline__ uint32_t code_exact(__half h, const GroupQ g, float mx)
{
    if (!g.fast) return code_int64<BITS>(__half2float(h), g.mn, mx);
    uint32_t q, qd;
    code_pair<BITS>(h, h, g, q, qd);
    return q & ((1u << BITS) - 1u);
}

// ------------------------------------------------------------ values (per token)
//
// Two threads per row: lane l works on row l & 15 of a 16-token block and on
// channels [64h, 64h + 64), h = l >> 4.  A block never crosses a (b, h) slice
// (blocks are numbered per slice; rows past S_q are computed and dropped), so
// it is two TMA tensor boxes of 16 rows x 64 channels, one per channel half,
// landing with the 128-byte swizzle: row r's 16-byte chunk c sits at chunk
// c ^ (r & 7) of its 128-byte line, and each quarter-warp of a 16-byte shared
// load touches eight distinct bank groups.  A per-warp 3-stage ring; a thread
// moves its 128 bytes to registers at once; the stage is refilled once the
// codes are done (the rare exact path reads it).  Per group: fp16 min/max (a 128-wide group combines the two
// halves by one shuffle), then the fast codes word by word; words go straight
// to global memory (the 16 rows x 2 halves of a block are contiguous there).

constexpr int VAL_WARPS = 20;
constexpr int VAL_STAGES = 2;
constexpr int VROWS = 16;
constexpr int VSTAGE_BYTES = VROWS * ROW_BYTES;  // two 2 KB swizzled boxes
// stages, mbarriers and the CTA's block counter
__host__ __device__ constexpr int val_smem_w(int warps) { return 1024 + warps * VAL_STAGES * (VSTAGE_BYTES + 8) + 16; }
__host__ __device__ constexpr int val_smem() { return val_smem_w(VAL_WARPS); }


__device__ __forceinline__ bool kivi_off(const KiviQuantParams &p, int b, int &off)
{
    off = 0;
    if (p.dst_off == nullptr) return true;
    off = __ldg(p.dst_off + b);
    if (off < 0 || off > p.S_dst - p.S_q || (off & (p.group - 1)) != 0) {
        atomicOr(&VQ_KIVI_ERR, (unsigned)VQ_DEVERR_BAD_OFFSET);
        return false;
    }
    return true;
}

__device__ __forceinline__ __half2 u2h2(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }

// The E codes of one values word, exactly (rare path), read from the staged
// block: base is the lane's 128-byte swizzled line, c0 the word's first chunk.
template <int BITS>
__device__ __noinline__ uint32_t values_word_exact(const unsigned char *base, int line, int c0, const GroupQ g,
                                                   float mx)
{
    constexpr int E = 32 / BITS;
    uint32_t word = 0u;
    for (int e = 0; e < E; ++e) {
        const __half h = *reinterpret_cast<const __half *>(base + swz128(line, c0 + e / 8) + 2 * (e % 8));
        word |= code_exact<BITS>(h, g, mx) << (e * BITS);
    }
    return word;
}

template <int BITS, int G, int WARPS>
__device__ __forceinline__ void kivi_values_body(const KiviQuantParams &p, int cta, int ncta)
{
    constexpr int E = 32 / BITS;           // codes per word
    constexpr int W = D * BITS / 32;       // words per row
    constexpr int WL = W / 2;              // words per thread
    constexpr int CPW = E / 8;             // 16-byte chunks per word
    constexpr int GL = G < 64 ? G : 64;    // group members held by one thread
    constexpr int NGL = 64 / GL;           // groups (or group halves) per thread
    constexpr int WPGL = WL / NGL;         // words per thread-group
    constexpr int CPG = GL / 8;            // chunks per thread-group
    constexpr int NGD = D / G;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    unsigned char *smem = smem_1k(smem_raw);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int rr = lane & 15, hh = lane >> 4;
    unsigned char *wbuf = smem + warp * (VAL_STAGES * VSTAGE_BYTES);
    uint64_t *bars_all = reinterpret_cast<uint64_t *>(smem + WARPS * VAL_STAGES * VSTAGE_BYTES);
    uint64_t *bars = bars_all + warp * VAL_STAGES;
    // the CTA takes the blocks [lo, hi) and its warps claim them one at a
    // time (a shared counter): warps whose blocks run slower take fewer, so
    // they finish together
    uint32_t *claimed = reinterpret_cast<uint32_t *>(bars_all + WARPS * VAL_STAGES);
    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < VAL_STAGES; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    if (threadIdx.x == 0) *claimed = 0u;
    __syncthreads();
    const uint64_t pol = l2_policy_evict_first();
    const int nsb = (p.S_q + VROWS - 1) / VROWS;  // blocks per (b, h) slice
    const int nblk = p.B * p.H * nsb;
    const int lo = (int)((long long)cta * nblk / ncta), hi = (int)((long long)(cta + 1) * nblk / ncta);
    auto claim = [&]() {
        int b = 0;
        if (lane == 0) b = lo + (int)atomicAdd(claimed, 1u);
        return __shfl_sync(FULL_MASK, b, 0);
    };

    auto issue = [&](int blk, int s) {
        if (lane == 0) {
            const int bh = fdiv(p.divBlk, blk), sb = blk - bh * nsb;
            mbar_arrive_expect_tx(&bars[s], (uint32_t)VSTAGE_BYTES);
            unsigned char *dst = wbuf + s * VSTAGE_BYTES;
            tma_load_3d(dst, &p.tmap, 0, sb * VROWS, bh, &bars[s], pol);
            tma_load_3d(dst + VSTAGE_BYTES / 2, &p.tmap, 64, sb * VROWS, bh, &bars[s], pol);
        }
    };
    // sb0, sb1: the blocks staged in stages 0 and 1 (claims are increasing,
    // and the stages are consumed in claim order)
    static_assert(VAL_STAGES == 2, "two stages per warp");
    int sb0 = claim();
    if (sb0 < hi) issue(sb0, 0);
    int sb1 = claim();
    if (sb1 < hi) issue(sb1, 1);
    for (int it = 0;; ++it) {
        const int s = it & 1;
        const int blk = s ? sb1 : sb0;
        if (blk >= hi) break;
        const bool ok = mbar_wait_bounded(&bars[s], (uint32_t)(it / VAL_STAGES) & 1u);
        if (!__all_sync(FULL_MASK, ok)) {
            if (lane == 0) atomicOr(&VQ_KIVI_ERR, (unsigned)VQ_DEVERR_WAIT_TIMEOUT);
            // the other stage's copy, if any, is still in flight
            const int it2 = it + 1;
            if ((s ? sb0 : sb1) < hi) (void)mbar_wait_bounded(&bars[it2 & 1], (uint32_t)(it2 >> 1) & 1u);
            return;
        }
        // this thread's 64 values to registers, then refill the stage
        uint4 c[8];
        const unsigned char *src = wbuf + s * VSTAGE_BYTES + hh * (VSTAGE_BYTES / 2);
#pragma unroll
        for (int i = 0; i < 8; ++i) c[i] = *reinterpret_cast<const uint4 *>(src + swz128(rr, i));

        const int bh = fdiv(p.divBlk, blk);
        const int s_ = (blk - bh * nsb) * VROWS + rr;
        size_t dr = 0;
        bool okrow = false;
        if (s_ < p.S_q) {
            int off;
            okrow = kivi_off(p, fdiv(p.divH, bh), off);
            dr = (size_t)bh * p.S_dst + off + s_;
        }
        uint32_t words[WL];
        __half scv[NGL], zrv[NGL];
#pragma unroll
        for (int jl = 0; jl < NGL; ++jl) {
            __half2 lo = u2h2(c[jl * CPG].x), hi = lo;
#pragma unroll
            for (int i = 0; i < CPG; ++i) {
                const uint4 q = c[jl * CPG + i];
                const __half2 a = __hmin2(__hmin2(u2h2(q.x), u2h2(q.y)), __hmin2(u2h2(q.z), u2h2(q.w)));
                const __half2 b = __hmax2(__hmax2(u2h2(q.x), u2h2(q.y)), __hmax2(u2h2(q.z), u2h2(q.w)));
                lo = __hmin2(lo, a);
                hi = __hmax2(hi, b);
            }
            float mn = fminf(__low2float(lo), __high2float(lo));
            float mx = fmaxf(__low2float(hi), __high2float(hi));
            if constexpr (G == 128) {
                mn = fminf(mn, __shfl_xor_sync(FULL_MASK, mn, 16));
                mx = fmaxf(mx, __shfl_xor_sync(FULL_MASK, mx, 16));
            }
            const GroupQ g = group_setup<BITS>(mn, mx);
            scv[jl] = g.scale_h;
            zrv[jl] = g.zero_h;
            const float2 f2 = make_float2(g.f, g.f), nf2 = make_float2(-g.f, -g.f);
#pragma unroll
            for (int w = 0; w < WPGL; ++w) {
                // two accumulators (first / second half of the word's codes)
                uint32_t alo = 0u, ahi = 0u, okw = 0xffffffffu;
#pragma unroll
                for (int ci = 0; ci < CPW; ++ci) {
                    const uint4 q = c[jl * CPG + w * CPW + ci];
                    const uint32_t u4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        uint32_t qa, qb;
                        code_pair_fast(__low2half(u2h2(u4[k])), __high2half(u2h2(u4[k])), mn, mn, f2, nf2,
                                       qa, qb, okw);
                        if (2 * (4 * ci + k) < E / 2) {
                            alo = __funnelshift_r(alo, qa, BITS);
                            alo = __funnelshift_r(alo, qb, BITS);
                        } else {
                            ahi = __funnelshift_r(ahi, qa, BITS);
                            ahi = __funnelshift_r(ahi, qb, BITS);
                        }
                    }
                }
                uint32_t word = (ahi & 0xffff0000u) | (alo >> 16);
                if (!(okw >> 31)) word = values_word_exact<BITS>(src, rr, jl * CPG + w * CPW, g, mx);
                words[jl * WPGL + w] = word;
            }
        }
        // the block is consumed: recycle the stage
        __syncwarp();
        fence_proxy_async_smem();
        {
            const int nb = claim();
            if (s)
                sb1 = nb;
            else
                sb0 = nb;
            if (nb < hi) issue(nb, s);
        }
        if (!okrow) continue;
        uint32_t *dst = p.packed + dr * W + hh * WL;
        if constexpr (WL == 2) {
            *reinterpret_cast<uint2 *>(dst) = make_uint2(words[0], words[1]);
        } else {
#pragma unroll
            for (int i = 0; i < WL / 4; ++i)
                reinterpret_cast<uint4 *>(dst)[i] = make_uint4(words[4 * i], words[4 * i + 1], words[4 * i + 2], words[4 * i + 3]);
        }
        __half *sc = static_cast<__half *>(p.scale) + dr * NGD;
        __half *zr = static_cast<__half *>(p.zero) + dr * NGD;
        if constexpr (G == 128) {
            if (hh == 0) {
                sc[0] = scv[0];
                zr[0] = zrv[0];
            }
        } else if constexpr (NGL == 2) {
            *reinterpret_cast<__half2 *>(sc + 2 * hh) = __halves2half2(scv[0], scv[1]);
            *reinterpret_cast<__half2 *>(zr + 2 * hh) = __halves2half2(zrv[0], zrv[1]);
        } else {
            sc[hh] = scv[0];
            zr[hh] = zrv[0];
        }
    }
}

// ------------------------------------------------------------ keys (per channel)
//
// One [G x 64] half-tile per warp step: channels [64c, 64c + 64) of the G
// tokens of a group, staged by one TMA tensor box (tokens past S arrive as
// zeros and are never used; tokens in [S_q, S) are ignored); lane l owns
// channels 2l and 2l + 1, so each token row of the tile is one conflict-free
// 32-bit load per lane and no cross-thread reduction is needed (the pages'
// "one thread, one whole group").  For G <= 64 the lane's 2G values move to
// registers in the min/max pass and the stage is refilled at once.  A word
// that holds a near-tie is redone inline by the exact FMA test (code_pair2);
// the rare group whose range fp32 does not hold is finished after the loop
// from global memory (no call inside the unrolled loop: a call site there
// costs the whole loop).  Codes of
// the two channels of a token run as one fp32 pair.  Each word row is stored
// as 8 bytes per lane (256 contiguous bytes per warp).

constexpr int KEY_SMEM_BUDGET = 220 * 1024;
constexpr int KEY_ROW = 128;  // bytes of one token row of a half-tile

// For G <= 64 the lane's tile column lives in registers after the min/max pass
// and the stage is refilled at once, so one stage per warp keeps a copy in
// flight during the codes; G = 128 reads the tile twice and double-buffers.
template <int G>
__host__ __device__ constexpr int key_stages()
{
    return G <= 64 ? 1 : 2;
}

template <int BITS, int G>
__host__ __device__ constexpr int key_warp_bytes()
{
    return key_stages<G>() * (G * KEY_ROW);
}

template <int BITS, int G>
__host__ __device__ constexpr int key_warps()
{
    return KEY_SMEM_BUDGET / (key_warp_bytes<BITS, G>() + 16) > 16 ? 16
                                                                      : KEY_SMEM_BUDGET / (key_warp_bytes<BITS, G>() + 16);
}

template <int BITS, int G>
__host__ __device__ constexpr int key_smem()
{
    return 1024 + key_warps<BITS, G>() * (key_warp_bytes<BITS, G>() + 16) + 16;  // + the CTA's tile counter
}

// Words of a tile column whose group range is not held exactly by fp32 and
// that hold a near-tie (rarely both): all codes of the flagged words again,
// exactly, from global memory.  xcol: channel 2l of the group's first token;
// dst: word row 0 of this lane's channel pair.
template <int BITS, int G>
__device__ __noinline__ void keys_words_slow(const __half *xcol, uint32_t *dst, uint32_t mask, int ntok,
                                             const GroupQ g0, const GroupQ g1, float mx0, float mx1)
{
    constexpr int E = 32 / BITS;
    for (int k = 0; k < G * BITS / 32; ++k) {
        if (!((mask >> k) & 1u)) continue;
        uint32_t w0 = 0u, w1 = 0u;
        for (int j = 0; j < E && k * E + j < ntok; ++j) {
            const __half2 h = *reinterpret_cast<const __half2 *>(xcol + (size_t)(k * E + j) * D);
            w0 |= code_exact<BITS>(__low2half(h), g0, mx0) << (j * BITS);
            w1 |= code_exact<BITS>(__high2half(h), g1, mx1) << (j * BITS);
        }
        *reinterpret_cast<uint2 *>(dst + (size_t)k * D) = make_uint2(w0, w1);
    }
}

template <int BITS, int G, int WARPS>
__device__ __forceinline__ void kivi_keys_body(const KiviQuantParams &p, int cta, int ncta)
{
    constexpr int KEY_WARPS = WARPS;
    constexpr int KEY_STAGES = key_stages<G>();
    constexpr int E = 32 / BITS;
    constexpr int WG = G * BITS / 32;  // words per channel per group
    constexpr int TILE = G * KEY_ROW;
    constexpr bool PRELOAD = G <= 64;
    constexpr int WBYTES = key_warp_bytes<BITS, G>();
    extern __shared__ __align__(128) unsigned char smem_raw[];
    unsigned char *smem = smem_1k(smem_raw);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    unsigned char *wbuf = smem + warp * WBYTES;
    uint64_t *bars_all = reinterpret_cast<uint64_t *>(smem + KEY_WARPS * WBYTES);
    uint64_t *bars = bars_all + warp * KEY_STAGES;
    // the CTA takes the half-tiles [lo, hi) and its warps claim them one at a
    // time (a shared counter), so that they finish together
    uint32_t *claimed = reinterpret_cast<uint32_t *>(bars_all + KEY_WARPS * KEY_STAGES);
    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < KEY_STAGES; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    if (threadIdx.x == 0) *claimed = 0u;
    __syncthreads();
    const uint64_t pol = l2_policy_evict_first();
    const int NG = (p.S_q + G - 1) / G;
    const int ntiles = p.B * p.H * NG * 2;
    const int lo = (int)((long long)cta * ntiles / ncta), hi = (int)((long long)(cta + 1) * ntiles / ncta);
    auto claim = [&]() {
        int t = 0;
        if (lane == 0) t = lo + (int)atomicAdd(claimed, 1u);
        return __shfl_sync(FULL_MASK, t, 0);
    };

    auto ntok_of = [&](int tile) {
        const int gi = tile >> 1;
        const int g = gi - fdiv(p.divBlk, gi) * NG;
        return min(G, p.S_q - g * G);
    };
    auto issue = [&](int tile, int s) {
        if (lane == 0) {
            const int gi = tile >> 1, chh = tile & 1;
            const int bh = fdiv(p.divBlk, gi), g = gi - bh * NG;
            mbar_arrive_expect_tx(&bars[s], (uint32_t)TILE);
            tma_load_3d(wbuf + s * TILE, &p.tmap, 64 * chh, g * G, bh, &bars[s], pol);
        }
    };
    // st0, st1: the half-tiles staged in stages 0 and 1 (claims are
    // increasing and consumed in claim order; one stage for G <= 64)
    static_assert(KEY_STAGES == 1 || KEY_STAGES == 2, "one or two stages per warp");
    int st0 = claim(), st1 = hi;
    if (st0 < hi) issue(st0, 0);
    if constexpr (KEY_STAGES == 2) {
        st1 = claim();
        if (st1 < hi) issue(st1, 1);
    }
    auto refill = [&](int s) {
        const int nt = claim();
        if (s)
            st1 = nt;
        else
            st0 = nt;
        if (nt < hi) issue(nt, s);
    };
    for (int it = 0;; ++it) {
        const int s = KEY_STAGES == 2 ? (it & 1) : 0;
        const int tile = s ? st1 : st0;
        if (tile >= hi) break;
        const bool ok = mbar_wait_bounded(&bars[s], (uint32_t)(it / KEY_STAGES) & 1u);
        if (!__all_sync(FULL_MASK, ok)) {
            if (lane == 0) atomicOr(&VQ_KIVI_ERR, (unsigned)VQ_DEVERR_WAIT_TIMEOUT);
            if (KEY_STAGES == 2 && (s ? st0 : st1) < hi) {
                const int it2 = it + 1;  // the other stage's copy is still in flight
                (void)mbar_wait_bounded(&bars[it2 & 1], (uint32_t)(it2 >> 1) & 1u);
            }
            return;
        }
        const uint32_t *col = reinterpret_cast<const uint32_t *>(wbuf + s * TILE) + lane;
        const int ntok = ntok_of(tile);
        const int gi = tile >> 1, chh = tile & 1;
        const int bh = fdiv(p.divBlk, gi), g = gi - bh * NG;

        // pass 1: min/max down the tokens (exact fp16); a ragged last group
        // is padded with its edge token, which leaves min/max unchanged
        uint32_t v[PRELOAD ? G : 1];
        __half2 lo, hi;
        if constexpr (PRELOAD) {
#pragma unroll
            for (int i = 0; i < G; ++i) v[i] = col[i * 32];
            if (ntok < G) {
                const uint32_t edge = col[(ntok - 1) * 32];
#pragma unroll
                for (int i = 0; i < G; ++i)
                    if (i >= ntok) v[i] = edge;
            }
            // the column is in registers: refill the stage now
            __syncwarp();
            fence_proxy_async_smem();
            refill(s);
            __half2 l2 = u2h2(v[0]), h2 = l2, l3 = u2h2(v[1]), h3 = l3;
#pragma unroll
            for (int i = 2; i < G; i += 2) {
                l2 = __hmin2(l2, u2h2(v[i]));
                h2 = __hmax2(h2, u2h2(v[i]));
                l3 = __hmin2(l3, u2h2(v[i + 1]));
                h3 = __hmax2(h3, u2h2(v[i + 1]));
            }
            lo = __hmin2(l2, l3);
            hi = __hmax2(h2, h3);
        } else {
            lo = u2h2(col[0]);
            hi = lo;
#pragma unroll 8
            for (int i = 1; i < ntok; ++i) {
                const __half2 a = u2h2(col[i * 32]);
                lo = __hmin2(lo, a);
                hi = __hmax2(hi, a);
            }
        }
        const float mx0 = __low2float(hi), mx1 = __high2float(hi);
        const GroupQ g0 = group_setup<BITS>(__low2float(lo), mx0);
        const GroupQ g1 = group_setup<BITS>(__high2float(lo), mx1);
        const float2 f2 = make_float2(g0.f, g1.f), nf2 = make_float2(-g0.f, -g1.f);
        int off;
        const bool okoff = kivi_off(p, fdiv(p.divH, bh), off);  // uniform across the warp
        const size_t gd = (size_t)bh * p.NG_dst + off / G + g;
        uint32_t *dst = p.packed + gd * WG * D + 64 * chh + 2 * lane;

        // pass 2: word row k holds tokens k*E .. k*E + E - 1 at shifts j*BITS
        const bool allfast = g0.fast && g1.fast;
        const float2 mn2 = make_float2(g0.mn, g1.mn), rr2 = make_float2(g0.rr, g1.rr);
        uint32_t slowmask = 0u;
#pragma unroll
        for (int k = 0; k < WG; ++k) {
            uint32_t a0 = 0u, b0 = 0u, a1 = 0u, b1 = 0u, okw = 0xffffffffu;
#pragma unroll
            for (int j = 0; j < E; ++j) {
                const int i = k * E + j;
                uint32_t u;
                if constexpr (PRELOAD) {
                    u = v[i];
                } else {
                    u = col[(i < ntok ? i : ntok - 1) * 32];
                }
                uint32_t q0, q1;
                code_pair_fast(__low2half(u2h2(u)), __high2half(u2h2(u)), g0.mn, g1.mn, f2, nf2, q0, q1,
                               okw);
                if (j < E / 2) {
                    a0 = __funnelshift_r(a0, q0, BITS);
                    a1 = __funnelshift_r(a1, q1, BITS);
                } else {
                    b0 = __funnelshift_r(b0, q0, BITS);
                    b1 = __funnelshift_r(b1, q1, BITS);
                }
            }
            if (!(okw >> 31)) {
                if (allfast) {
                    // a near-tie in the word: exact codes for all of it
                    a0 = b0 = a1 = b1 = 0u;
#pragma unroll
                    for (int j = 0; j < E; ++j) {
                        const int i = k * E + j;
                        uint32_t u;
                        if constexpr (PRELOAD) {
                            u = v[i];
                        } else {
                            u = col[(i < ntok ? i : ntok - 1) * 32];
                        }
                        uint32_t q0, q1;
                        code_pair2<BITS>(__low2half(u2h2(u)), __high2half(u2h2(u)), mn2, f2, rr2, q0, q1);
                        if (j < E / 2) {
                            a0 = __funnelshift_r(a0, q0, BITS);
                            a1 = __funnelshift_r(a1, q1, BITS);
                        } else {
                            b0 = __funnelshift_r(b0, q0, BITS);
                            b1 = __funnelshift_r(b1, q1, BITS);
                        }
                    }
                } else {
                    slowmask |= 1u << k;
                }
            }
            uint32_t w0 = (b0 & 0xffff0000u) | (a0 >> 16);
            uint32_t w1 = (b1 & 0xffff0000u) | (a1 >> 16);
            const int nvalid = ntok - k * E;  // tokens of this word that exist
            if (nvalid < E) {  // slots past the last token hold 0
                const uint32_t m = nvalid <= 0 ? 0u : (0xffffffffu >> (32 - nvalid * BITS));
                w0 &= m;
                w1 &= m;
            }
            if (okoff) *reinterpret_cast<uint2 *>(dst + (size_t)k * D) = make_uint2(w0, w1);
        }
        if (slowmask != 0u && okoff)
            keys_words_slow<BITS, G>(static_cast<const __half *>(p.x) + ((size_t)bh * p.S + (size_t)g * G) * D +
                                         64 * chh + 2 * lane,
                                     dst, slowmask, ntok, g0, g1, mx0, mx1);
        if constexpr (!PRELOAD) {
            // the tile is consumed: recycle the stage
            __syncwarp();
            fence_proxy_async_smem();
            refill(s);
        }
        if (!okoff) continue;
        *reinterpret_cast<__half2 *>(static_cast<__half *>(p.scale) + gd * D + 64 * chh + 2 * lane) =
            __halves2half2(g0.scale_h, g1.scale_h);
        *reinterpret_cast<__half2 *>(static_cast<__half *>(p.zero) + gd * D + 64 * chh + 2 * lane) =
            __halves2half2(g0.zero_h, g1.zero_h);
    }
}

}  // namespace
}  // namespace vq
