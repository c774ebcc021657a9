// kivi.cu - KIVI asymmetric min/max group quantize+pack and unpack+dequant
// for sm_103a.
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
// Values (per token): one row per thread, rows staged by per-row bulk copies
// into a per-warp 3-stage ring (as the RVQ encoder).  Keys (per channel): one
// [G x 128] tile (contiguous in memory) per warp per step, staged by a single
// bulk copy; lane l owns channels 4l..4l+3 and walks the G tokens, so no
// cross-thread reduction is needed (the pages' "one thread, one whole group").
#include <cuda_fp16.h>

#include "device_common.cuh"
#include "launch.h"

namespace vq {

VQ_DEFINE_ERROR_WORD(g_kivi_err);

namespace {

constexpr int D = 128;
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
__device__ __forceinline__ void code_pair(__half a, __half b, const GroupQ &g, uint32_t &qa,
                                          uint32_t &qb)
{
    constexpr float C = (float)((1 << BITS) - 1);
    const float2 A = make_float2(add_f16_f32(a, -g.mn), add_f16_f32(b, -g.mn));
    const float2 tm = __ffma2_rn(A, make_float2(g.f, g.f), make_float2(MAGIC1, MAGIC1));
    const float2 r = __fadd2_rn(tm, make_float2(-MAGIC1, -MAGIC1));
    const float2 ca = __fmul2_rn(A, make_float2(C, C));
    const float2 u = __ffma2_rn(r, make_float2(-g.rr, -g.rr), ca);
    const float h = 0.5f * g.rr;
    const float2 zl = __fadd2_rn(u, make_float2(h, h));
    const float2 zr = __fadd2_rn(u, make_float2(-h, -h));
    const float2 st = __fadd2_rn(make_float2(step_half(zl.x), step_half(zl.y)),
                                 make_float2(step_half(zr.x), step_half(zr.y)));
    const float2 qm = __fadd2_rn(tm, st);  // MAGIC + q, ties to even
    qa = __float_as_uint(qm.x);
    qb = __float_as_uint(qm.y);
}

// fp16(q*s + z) rounded once from the exact value: q*s is exact in fp32, the
// sum is carried as a rounded value plus its exact error, and a non-zero error
// is folded in as a sticky bit (round-to-odd) before the final fp16 rounding.
__device__ __forceinline__ __half recon_exact(uint32_t q, float s, float z)
{
    const float p = (float)q * s;
    float sum, err;
    two_sum(p, z, sum, err);
    if (err != 0.0f) {
        uint32_t b = __float_as_uint(sum);
        if ((err < 0.0f) != (sum < 0.0f)) b -= 1u;  // truncate toward zero
        b |= 1u;                                     // sticky
        sum = __uint_as_float(b);
    }
    return __float2half_rn(sum);
}

// True when q*s + z is exact in fp32 for every q in [0, C]: the sum then
// needs no more than 24 significant bits.  s and z are fp16 values; their
// quanta are ulp16 (2^-24 for subnormals).
__device__ __forceinline__ float ulp16_of(float x)
{
    int e = ((__float_as_int(x) >> 23) & 0xff) - 127;
    e = e < -14 ? -14 : e;
    return __int_as_float((e - 10 + 127) << 23);
}

template <int BITS>
__device__ __forceinline__ bool group_sum_exact(float s, float z)
{
    constexpr float C = (float)((1 << BITS) - 1);
    if (s == 0.0f || z == 0.0f) return true;
    const float q = fminf(ulp16_of(s), ulp16_of(z));
    return fabsf(z) + C * s < 8388608.0f * q;  // 2^23 quanta: one bit of headroom
}

// ------------------------------------------------------------ values (per token)
//
// One row per thread, 32-row blocks per warp.  Rows arrive by per-row bulk
// copies (rows skip the residual window, so a block need not be contiguous)
// into a 3-stage ring at a 272-byte stride.  Per group: fp16 min/max, then a
// rolled loop over the group's output words; words and (scale, zero) are
// staged in shared memory and written out coalesced.

constexpr int VAL_WARPS = 8;
constexpr int VAL_STAGES = 3;
constexpr int ROW_BYTES = D * 2;
constexpr int ROW_STRIDE = ROW_BYTES + 16;
constexpr int VSTAGE_BYTES = 32 * ROW_STRIDE;
__host__ __device__ constexpr int val_words(int bits) { return D * bits / 32; }
__host__ __device__ constexpr int val_warp_bytes(int bits, int G)
{
    return VAL_STAGES * VSTAGE_BYTES + 32 * (val_words(bits) + 1) * 4 + 32 * (D / G) * 4;
}
__host__ __device__ constexpr int val_smem(int bits, int G)
{
    return VAL_WARPS * (val_warp_bytes(bits, G) + VAL_STAGES * 8);
}

__device__ __forceinline__ bool kivi_off(const KiviQuantParams &p, int b, int &off)
{
    off = 0;
    if (p.dst_off == nullptr) return true;
    off = __ldg(p.dst_off + b);
    if (off < 0 || off > p.S_dst - p.S_q || (off % p.group) != 0) {
        atomicOr(&g_kivi_err, (unsigned)VQ_DEVERR_BAD_OFFSET);
        return false;
    }
    return true;
}

__device__ __forceinline__ uint32_t h2bits(__half h) { return (uint32_t)__half_as_ushort(h); }

template <int BITS, int G>
__global__ void __launch_bounds__(VAL_WARPS * 32, 1)
    kivi_values_kernel(const __grid_constant__ KiviQuantParams p)
{
    constexpr int E = 32 / BITS;
    constexpr int W = D * BITS / 32;
    constexpr int NGD = D / G;
    constexpr int WPG = G * BITS / 32;  // words per group
    constexpr int WB = val_warp_bytes(BITS, G);
    extern __shared__ __align__(128) unsigned char smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    unsigned char *wbuf = smem + warp * WB;
    uint32_t *ow = reinterpret_cast<uint32_t *>(wbuf + VAL_STAGES * VSTAGE_BYTES);
    uint32_t *osz = ow + 32 * (W + 1);  // scale | zero << 16, per row and group
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + VAL_WARPS * WB) + warp * VAL_STAGES;
    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < VAL_STAGES; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    __syncwarp();
    const uint64_t pol = l2_policy_evict_first();
    const int N = p.B * p.H * p.S_q;
    const int nblk = (N + 31) >> 5;
    const int gw = blockIdx.x * VAL_WARPS + warp;
    const int tw = gridDim.x * VAL_WARPS;
    const __half *x = static_cast<const __half *>(p.x);

    auto issue = [&](int blk, int s) {
        const int r0 = blk << 5;
        const int nrows = min(32, N - r0);
        if (lane == 0) mbar_arrive_expect_tx(&bars[s], (uint32_t)(nrows * ROW_BYTES));
        if (lane < nrows) {
            const int r = r0 + lane;
            const int bh = r / p.S_q, s_ = r - bh * p.S_q;
            bulk_g2s(wbuf + s * VSTAGE_BYTES + lane * ROW_STRIDE,
                     x + ((size_t)bh * p.S + s_) * D, ROW_BYTES, &bars[s], pol);
        }
    };
#pragma unroll
    for (int s = 0; s < VAL_STAGES; ++s) {
        const int blk = gw + s * tw;
        if (blk < nblk) issue(blk, s);
    }
    for (int it = 0;; ++it) {
        const int blk = gw + it * tw;
        if (blk >= nblk) break;
        const int s = it % VAL_STAGES;
        const bool ok = mbar_wait_bounded(&bars[s], (uint32_t)(it / VAL_STAGES) & 1u);
        if (!__all_sync(FULL_MASK, ok)) {
            if (lane == 0) atomicOr(&g_kivi_err, (unsigned)VQ_DEVERR_WAIT_TIMEOUT);
            for (int k = 1; k < VAL_STAGES; ++k) {
                const int it2 = it + k;
                if (gw + it2 * tw < nblk)
                    (void)mbar_wait_bounded(&bars[it2 % VAL_STAGES], (uint32_t)(it2 / VAL_STAGES) & 1u);
            }
            return;
        }
        const int row = (blk << 5) + lane;
        const __half *rh = reinterpret_cast<const __half *>(wbuf + s * VSTAGE_BYTES + lane * ROW_STRIDE);
#pragma unroll 1
        for (int j = 0; j < NGD; ++j) {
            const uint4 *gp = reinterpret_cast<const uint4 *>(rh + j * G);
            uint4 c0 = gp[0];
            __half2 lo = __hmin2(__hmin2(*reinterpret_cast<__half2 *>(&c0.x), *reinterpret_cast<__half2 *>(&c0.y)),
                                 __hmin2(*reinterpret_cast<__half2 *>(&c0.z), *reinterpret_cast<__half2 *>(&c0.w)));
            __half2 hi = __hmax2(__hmax2(*reinterpret_cast<__half2 *>(&c0.x), *reinterpret_cast<__half2 *>(&c0.y)),
                                 __hmax2(*reinterpret_cast<__half2 *>(&c0.z), *reinterpret_cast<__half2 *>(&c0.w)));
#pragma unroll
            for (int i = 1; i < G / 8; ++i) {
                uint4 c = gp[i];
                lo = __hmin2(lo, __hmin2(__hmin2(*reinterpret_cast<__half2 *>(&c.x), *reinterpret_cast<__half2 *>(&c.y)),
                                         __hmin2(*reinterpret_cast<__half2 *>(&c.z), *reinterpret_cast<__half2 *>(&c.w))));
                hi = __hmax2(hi, __hmax2(__hmax2(*reinterpret_cast<__half2 *>(&c.x), *reinterpret_cast<__half2 *>(&c.y)),
                                         __hmax2(*reinterpret_cast<__half2 *>(&c.z), *reinterpret_cast<__half2 *>(&c.w))));
            }
            const float mn = fminf(__low2float(lo), __high2float(lo));
            const float mx = fmaxf(__low2float(hi), __high2float(hi));
            const GroupQ g = group_setup<BITS>(mn, mx);
            osz[lane * NGD + j] = h2bits(g.scale_h) | (h2bits(g.zero_h) << 16);
#pragma unroll 1
            for (int w = 0; w < WPG; ++w) {
                const uint4 *wp = gp + w * (E / 8);
                uint32_t word = 0u;
                if (g.fast) {
                    // two accumulators (first and second half of the word's
                    // codes) halve the dependent chain of funnel shifts
                    uint32_t lo = 0u, hi = 0u;
#pragma unroll
                    for (int i = 0; i < E / 8; ++i) {
                        uint4 c = wp[i];
                        const __half2 *hh = reinterpret_cast<const __half2 *>(&c);
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            uint32_t qa, qb;
                            code_pair<BITS>(__low2half(hh[k]), __high2half(hh[k]), g, qa, qb);
                            if (i < E / 16 || (E == 8 && k < 2)) {
                                lo = __funnelshift_r(lo, qa, BITS);
                                lo = __funnelshift_r(lo, qb, BITS);
                            } else {
                                hi = __funnelshift_r(hi, qa, BITS);
                                hi = __funnelshift_r(hi, qb, BITS);
                            }
                        }
                    }
                    word = (hi & 0xffff0000u) | (lo >> 16);
                } else {  // rare: a range that fp32 does not hold exactly
                    for (int e = 0; e < E; ++e)
                        word |= code_int64<BITS>(__half2float(rh[j * G + w * E + e]), mn, mx) << (e * BITS);
                }
                ow[lane * (W + 1) + j * WPG + w] = word;
            }
        }
        // the block is in registers / staging: recycle the stage
        __syncwarp();
        fence_proxy_async_smem();
        {
            const int nb = blk + VAL_STAGES * tw;
            if (nb < nblk) issue(nb, s);
        }
        // coalesced write-out
        int dr32 = 0;
        bool okrow = false;
        if (row < N) {
            const int bh = row / p.S_q, s_ = row - bh * p.S_q;
            int off;
            okrow = kivi_off(p, bh / p.H, off);
            dr32 = bh * p.S_dst + off + s_;
        }
#pragma unroll
        for (int i = 0; i < W; ++i) {
            const int idx = i * 32 + lane;
            const int r = idx / W, w = idx % W;
            const int dr = __shfl_sync(FULL_MASK, dr32, r);
            if (__shfl_sync(FULL_MASK, okrow ? 1 : 0, r)) p.packed[(size_t)dr * W + w] = ow[r * (W + 1) + w];
        }
        __half *sc = static_cast<__half *>(p.scale);
        __half *zr = static_cast<__half *>(p.zero);
#pragma unroll
        for (int i = 0; i < NGD; ++i) {
            const int idx = i * 32 + lane;
            const int r = idx / NGD, j = idx % NGD;
            const int dr = __shfl_sync(FULL_MASK, dr32, r);
            if (__shfl_sync(FULL_MASK, okrow ? 1 : 0, r)) {
                const uint32_t v = osz[r * NGD + j];
                sc[(size_t)dr * NGD + j] = __ushort_as_half((unsigned short)(v & 0xffffu));
                zr[(size_t)dr * NGD + j] = __ushort_as_half((unsigned short)(v >> 16));
            }
        }
        __syncwarp();
    }
}

// ------------------------------------------------------------ keys (per channel)
//
// One [G x 128] tile (contiguous in memory) per warp per step, one bulk copy;
// lane l owns channels 4l..4l+3.  Pass 1: fp16 min/max down the tokens.
// Pass 2: a rolled loop over the group's word rows; each step packs E tokens
// of the lane's four channels into four words and stores them as one 16-byte
// write (512 contiguous bytes per warp).

constexpr int KEY_STAGES = 2;
constexpr int KEY_SMEM_BUDGET = 192 * 1024;

// Warps per CTA for key tiles of G tokens: as many 2-stage rings as fit.
template <int G>
__host__ __device__ constexpr int key_warps()
{
    return KEY_SMEM_BUDGET / (KEY_STAGES * G * ROW_BYTES) > 12 ? 12
                                                                 : KEY_SMEM_BUDGET / (KEY_STAGES * G * ROW_BYTES);
}

template <int G>
__host__ __device__ constexpr int key_smem()
{
    return key_warps<G>() * KEY_STAGES * (G * ROW_BYTES + 8);
}

template <int BITS, int G>
__global__ void __launch_bounds__(key_warps<G>() * 32, 1)
    kivi_keys_kernel(const __grid_constant__ KiviQuantParams p)
{
    constexpr int KEY_WARPS = key_warps<G>();
    constexpr int E = 32 / BITS;
    constexpr int WG = G * BITS / 32;  // words per channel per group
    constexpr int TILE = G * ROW_BYTES;
    extern __shared__ __align__(128) unsigned char smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    unsigned char *wbuf = smem + warp * (KEY_STAGES * TILE);
    uint64_t *bars =
        reinterpret_cast<uint64_t *>(smem + KEY_WARPS * KEY_STAGES * TILE) + warp * KEY_STAGES;
    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < KEY_STAGES; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    __syncwarp();
    const uint64_t pol = l2_policy_evict_first();
    const int NG = (p.S_q + G - 1) / G;
    const int ntiles = p.B * p.H * NG;
    const int gw = blockIdx.x * KEY_WARPS + warp;
    const int tw = gridDim.x * KEY_WARPS;
    const __half *x = static_cast<const __half *>(p.x);

    auto ntok_of = [&](int tile) {
        const int g = tile % NG;
        return min(G, p.S_q - g * G);
    };
    auto issue = [&](int tile, int s) {
        if (lane == 0) {
            const int bh = tile / NG, g = tile - bh * NG;
            const uint32_t bytes = (uint32_t)(ntok_of(tile) * ROW_BYTES);
            mbar_arrive_expect_tx(&bars[s], bytes);
            bulk_g2s(wbuf + s * TILE, x + ((size_t)bh * p.S + (size_t)g * G) * D, bytes, &bars[s], pol);
        }
    };
#pragma unroll
    for (int s = 0; s < KEY_STAGES; ++s) {
        const int t = gw + s * tw;
        if (t < ntiles) issue(t, s);
    }
    for (int it = 0;; ++it) {
        const int tile = gw + it * tw;
        if (tile >= ntiles) break;
        const int s = it % KEY_STAGES;
        const bool ok = mbar_wait_bounded(&bars[s], (uint32_t)(it / KEY_STAGES) & 1u);
        if (!__all_sync(FULL_MASK, ok)) {
            if (lane == 0) atomicOr(&g_kivi_err, (unsigned)VQ_DEVERR_WAIT_TIMEOUT);
            for (int k = 1; k < KEY_STAGES; ++k) {
                const int it2 = it + k;
                if (gw + it2 * tw < ntiles)
                    (void)mbar_wait_bounded(&bars[it2 % KEY_STAGES], (uint32_t)(it2 / KEY_STAGES) & 1u);
            }
            return;
        }
        const unsigned char *tb = wbuf + s * TILE;
        const int ntok = ntok_of(tile);
        const int bh = tile / NG, g = tile - bh * NG;
        // pass 1: per-channel min/max over the group's tokens (exact fp16)
        const uint2 *col = reinterpret_cast<const uint2 *>(tb) + lane;  // channels 4l..4l+3
        uint2 r0 = col[0];
        __half2 lo0 = *reinterpret_cast<__half2 *>(&r0.x), lo1 = *reinterpret_cast<__half2 *>(&r0.y);
        __half2 hi0 = lo0, hi1 = lo1;
#pragma unroll 8
        for (int i = 1; i < ntok; ++i) {
            uint2 r = col[i * (ROW_BYTES / 8)];
            const __half2 a = *reinterpret_cast<__half2 *>(&r.x), b = *reinterpret_cast<__half2 *>(&r.y);
            lo0 = __hmin2(lo0, a); hi0 = __hmax2(hi0, a);
            lo1 = __hmin2(lo1, b); hi1 = __hmax2(hi1, b);
        }
        const float mxv[4] = {__low2float(hi0), __high2float(hi0), __low2float(hi1), __high2float(hi1)};
        GroupQ gq[4];
        gq[0] = group_setup<BITS>(__low2float(lo0), mxv[0]);
        gq[1] = group_setup<BITS>(__high2float(lo0), mxv[1]);
        gq[2] = group_setup<BITS>(__low2float(lo1), mxv[2]);
        gq[3] = group_setup<BITS>(__high2float(lo1), mxv[3]);
        int off;
        const bool okoff = kivi_off(p, bh / p.H, off);  // uniform across the warp
        const size_t gd = (size_t)bh * p.NG_dst + off / G + g;
        // pass 2: word row k holds tokens k*E .. k*E + E - 1 at shifts j*BITS
        const __half *tokh = reinterpret_cast<const __half *>(tb);
        const bool allfast = gq[0].fast && gq[1].fast && gq[2].fast && gq[3].fast;
#pragma unroll 1
        for (int k = 0; k < WG; ++k) {
            uint32_t w0 = 0u, w1 = 0u, w2 = 0u, w3 = 0u;
            if (allfast) {
#pragma unroll
                for (int j = 0; j < E; j += 2) {
                    const int i = k * E + j;
                    uint32_t c0a = 0, c0b = 0, c1a = 0, c1b = 0, c2a = 0, c2b = 0, c3a = 0, c3b = 0;
                    if (i < ntok) {
                        uint2 ra = col[i * (ROW_BYTES / 8)];
                        uint2 rb = (i + 1 < ntok) ? col[(i + 1) * (ROW_BYTES / 8)] : ra;
                        const __half2 a01 = *reinterpret_cast<__half2 *>(&ra.x), a23 = *reinterpret_cast<__half2 *>(&ra.y);
                        const __half2 b01 = *reinterpret_cast<__half2 *>(&rb.x), b23 = *reinterpret_cast<__half2 *>(&rb.y);
                        code_pair<BITS>(__low2half(a01), __low2half(b01), gq[0], c0a, c0b);
                        code_pair<BITS>(__high2half(a01), __high2half(b01), gq[1], c1a, c1b);
                        code_pair<BITS>(__low2half(a23), __low2half(b23), gq[2], c2a, c2b);
                        code_pair<BITS>(__high2half(a23), __high2half(b23), gq[3], c3a, c3b);
                        if (i + 1 >= ntok) c0b = c1b = c2b = c3b = 0u;
                    }
                    w0 = __funnelshift_r(__funnelshift_r(w0, c0a, BITS), c0b, BITS);
                    w1 = __funnelshift_r(__funnelshift_r(w1, c1a, BITS), c1b, BITS);
                    w2 = __funnelshift_r(__funnelshift_r(w2, c2a, BITS), c2b, BITS);
                    w3 = __funnelshift_r(__funnelshift_r(w3, c3a, BITS), c3b, BITS);
                }
            } else {  // rare: some channel's range is not held exactly by fp32
                uint32_t rw[4] = {0u, 0u, 0u, 0u};
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    for (int j = 0; j < E; ++j) {
                        const int i = k * E + j;
                        if (i >= ntok) break;
                        const float xv = __half2float(tokh[i * D + 4 * lane + c]);
                        uint32_t q, qdummy;
                        if (gq[c].fast) {
                            code_pair<BITS>(__float2half_rn(xv), __float2half_rn(xv), gq[c], q, qdummy);
                            q &= (1u << BITS) - 1u;
                        } else {
                            q = code_int64<BITS>(xv, gq[c].mn, mxv[c]);
                        }
                        rw[c] |= q << (j * BITS);
                    }
                }
                w0 = rw[0]; w1 = rw[1]; w2 = rw[2]; w3 = rw[3];
            }
            if (okoff)
                *reinterpret_cast<uint4 *>(p.packed + (gd * WG + k) * D + 4 * lane) = make_uint4(w0, w1, w2, w3);
        }
        // the tile is consumed: recycle the stage
        __syncwarp();
        fence_proxy_async_smem();
        {
            const int nt = tile + KEY_STAGES * tw;
            if (nt < ntiles) issue(nt, s);
        }
        if (!okoff) continue;
        __half2 s01 = __halves2half2(gq[0].scale_h, gq[1].scale_h);
        __half2 s23 = __halves2half2(gq[2].scale_h, gq[3].scale_h);
        __half2 z01 = __halves2half2(gq[0].zero_h, gq[1].zero_h);
        __half2 z23 = __halves2half2(gq[2].zero_h, gq[3].zero_h);
        *reinterpret_cast<uint2 *>(static_cast<__half *>(p.scale) + gd * D + 4 * lane) =
            make_uint2(*reinterpret_cast<uint32_t *>(&s01), *reinterpret_cast<uint32_t *>(&s23));
        *reinterpret_cast<uint2 *>(static_cast<__half *>(p.zero) + gd * D + 4 * lane) =
            make_uint2(*reinterpret_cast<uint32_t *>(&z01), *reinterpret_cast<uint32_t *>(&z23));
    }
}

// ------------------------------------------------------------ dequant

constexpr int DQ_THREADS = 256;

// Values: one row per thread; each row's words arrive by a per-row bulk copy
// into a 3-stage ring (slots padded for conflict-free 16-byte reads); the fp16
// row is staged in shared memory and written out coalesced.
constexpr int VDQ_WARPS = 8;
constexpr int VDQ_STAGES = 3;
__host__ __device__ constexpr int vdq_slot(int bits) { return (D * bits / 32) * 4 + 16 > 48 ? (D * bits / 32) * 4 + 16 : 48; }
__host__ __device__ constexpr int vdq_warp_bytes(int bits) { return VDQ_STAGES * 32 * vdq_slot(bits) + 32 * ROW_STRIDE; }
__host__ __device__ constexpr int vdq_smem(int bits) { return VDQ_WARPS * (vdq_warp_bytes(bits) + VDQ_STAGES * 8); }

// One group of a row whose q*s + z is not exact in fp32 (rare): every element
// goes through recon_exact.  wg: the group's words; out: its 16-byte output
// chunks in the staging row.
template <int BITS, int G>
__device__ __noinline__ void vdq_group_exact(const uint32_t *wg, float s, float z, uint4 *out)
{
    constexpr int E = 32 / BITS;
    constexpr uint32_t MASK = (1u << BITS) - 1u;
    for (int c = 0; c < G / 8; ++c) {
        uint32_t o[4];
        for (int j = 0; j < 4; ++j) {
            const int e = 8 * c + 2 * j;
            const uint32_t q0 = (wg[e / E] >> ((e % E) * BITS)) & MASK;
            const uint32_t q1 = (wg[(e + 1) / E] >> (((e + 1) % E) * BITS)) & MASK;
            const __half2 hv = __halves2half2(recon_exact(q0, s, z), recon_exact(q1, s, z));
            o[j] = *reinterpret_cast<const uint32_t *>(&hv);
        }
        out[c] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

template <int BITS, int G>
__global__ void __launch_bounds__(VDQ_WARPS * 32, 1) kivi_values_dequant_kernel(const __grid_constant__ KiviDequantParams p)
{
    constexpr int E = 32 / BITS;
    constexpr int W = D * BITS / 32;
    constexpr int NGD = D / G;
    constexpr int WPG = G * BITS / 32;
    constexpr uint32_t MASK = (1u << BITS) - 1u;
    constexpr int SLOT = vdq_slot(BITS);
    constexpr int WB = vdq_warp_bytes(BITS);
    extern __shared__ __align__(128) unsigned char smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    unsigned char *wbuf = smem + warp * WB;
    unsigned char *obuf = wbuf + VDQ_STAGES * 32 * SLOT;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + VDQ_WARPS * WB) + warp * VDQ_STAGES;
    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < VDQ_STAGES; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    __syncwarp();
    const uint64_t pol = l2_policy_evict_first();
    const int N = p.BH * p.S_q;
    const int nblk = (N + 31) >> 5;
    const int gw = blockIdx.x * VDQ_WARPS + warp;
    const int tw = gridDim.x * VDQ_WARPS;
    auto issue = [&](int blk, int s) {
        const int r0 = blk << 5;
        const int nrows = min(32, N - r0);
        if (lane == 0) mbar_arrive_expect_tx(&bars[s], (uint32_t)(nrows * W * 4));
        if (lane < nrows)
            bulk_g2s(wbuf + s * 32 * SLOT + lane * SLOT, p.packed + (size_t)(r0 + lane) * W, W * 4, &bars[s], pol);
    };
#pragma unroll
    for (int s = 0; s < VDQ_STAGES; ++s) {
        const int blk = gw + s * tw;
        if (blk < nblk) issue(blk, s);
    }
    const __half *scp = static_cast<const __half *>(p.scale);
    const __half *zrp = static_cast<const __half *>(p.zero);
    // scale/zero of this lane's row, loaded one block ahead
    __half sh[NGD], zh[NGD];
    auto load_sz = [&](int blk) {
        const int row = (blk << 5) + lane;
#pragma unroll
        for (int j = 0; j < NGD; ++j) {
            sh[j] = (blk < nblk && row < N) ? scp[(size_t)row * NGD + j] : __float2half_rn(0.0f);
            zh[j] = (blk < nblk && row < N) ? zrp[(size_t)row * NGD + j] : __float2half_rn(0.0f);
        }
    };
    load_sz(gw);
    for (int it = 0;; ++it) {
        const int blk = gw + it * tw;
        if (blk >= nblk) break;
        const int s = it % VDQ_STAGES;
        float sf[NGD], zf[NGD];
#pragma unroll
        for (int j = 0; j < NGD; ++j) {
            sf[j] = __half2float(sh[j]);
            zf[j] = __half2float(zh[j]);
        }
        load_sz(blk + tw);
        const bool ok = mbar_wait_bounded(&bars[s], (uint32_t)(it / VDQ_STAGES) & 1u);
        if (!__all_sync(FULL_MASK, ok)) {
            if (lane == 0) atomicOr(&g_kivi_err, (unsigned)VQ_DEVERR_WAIT_TIMEOUT);
            for (int k = 1; k < VDQ_STAGES; ++k) {
                const int it2 = it + k;
                if (gw + it2 * tw < nblk)
                    (void)mbar_wait_bounded(&bars[it2 % VDQ_STAGES], (uint32_t)(it2 / VDQ_STAGES) & 1u);
            }
            return;
        }
        const uint32_t *wrow = reinterpret_cast<const uint32_t *>(wbuf + s * 32 * SLOT + lane * SLOT);
        uint4 *orow = reinterpret_cast<uint4 *>(obuf + lane * ROW_STRIDE);
#pragma unroll
        for (int j = 0; j < NGD; ++j) {
            if (group_sum_exact<BITS>(sf[j], zf[j])) {
                uint32_t wg[WPG];
#pragma unroll
                for (int i = 0; i < WPG; i += 4) {
                    if constexpr (WPG >= 4) {
                        const uint4 a = *reinterpret_cast<const uint4 *>(wrow + j * WPG + i);
                        wg[i] = a.x; wg[i + 1] = a.y; wg[i + 2] = a.z; wg[i + 3] = a.w;
                    }
                }
                if constexpr (WPG < 4) {
#pragma unroll
                    for (int i = 0; i < WPG; ++i) wg[i] = wrow[j * WPG + i];
                }
#pragma unroll
                for (int c = 0; c < G / 8; ++c) {
                    uint32_t o[4];
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        const int e = 8 * c + 2 * jj;
                        const uint32_t q0 = (wg[e / E] >> ((e % E) * BITS)) & MASK;
                        const uint32_t q1 = (wg[(e + 1) / E] >> (((e + 1) % E) * BITS)) & MASK;
                        const __half2 hv = __floats2half2_rn(fmaf((float)q0, sf[j], zf[j]), fmaf((float)q1, sf[j], zf[j]));
                        o[jj] = *reinterpret_cast<const uint32_t *>(&hv);
                    }
                    orow[j * (G / 8) + c] = make_uint4(o[0], o[1], o[2], o[3]);
                }
            } else {
                vdq_group_exact<BITS, G>(wrow + j * WPG, sf[j], zf[j], orow + j * (G / 8));
            }
        }
        __syncwarp();
        fence_proxy_async_smem();
        {
            const int nb = blk + VDQ_STAGES * tw;
            if (nb < nblk) issue(nb, s);
        }
        const int nrows = min(32, N - (blk << 5));
        uint4 *gout = reinterpret_cast<uint4 *>(static_cast<__half *>(p.out) + (size_t)(blk << 5) * D);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int idx = i * 32 + lane;
            const int r = idx >> 4, c = idx & 15;
            if (r < nrows) gout[idx] = *reinterpret_cast<const uint4 *>(obuf + r * ROW_STRIDE + c * 16);
        }
        __syncwarp();
    }
}

template <int BITS, int G>
__global__ void __launch_bounds__(DQ_THREADS) kivi_keys_dequant_kernel(const __grid_constant__ KiviDequantParams p)
{
    constexpr int E = 32 / BITS;
    constexpr int WG = G * BITS / 32;
    constexpr uint32_t MASK = (1u << BITS) - 1u;
    const int lane = threadIdx.x & 31;
    const int wpb = DQ_THREADS / 32;
    const int ntiles = p.BH * p.NG;
    for (int tile = blockIdx.x * wpb + (threadIdx.x >> 5); tile < ntiles; tile += gridDim.x * wpb) {
        const int bh = tile / p.NG, g = tile - bh * p.NG;
        const int ntok = min(G, p.S_q - g * G);
        const uint2 sraw = __ldg(reinterpret_cast<const uint2 *>(static_cast<const __half *>(p.scale) + (size_t)tile * D + 4 * lane));
        const uint2 zraw = __ldg(reinterpret_cast<const uint2 *>(static_cast<const __half *>(p.zero) + (size_t)tile * D + 4 * lane));
        const __half *sh = reinterpret_cast<const __half *>(&sraw);
        const __half *zh = reinterpret_cast<const __half *>(&zraw);
        float s[4], z[4];
        bool all_exact = true;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            s[j] = __half2float(sh[j]);
            z[j] = __half2float(zh[j]);
            all_exact &= group_sum_exact<BITS>(s[j], z[j]);
        }
        for (int k = 0; k < WG; ++k) {
            const uint4 wv = __ldg(reinterpret_cast<const uint4 *>(p.packed + ((size_t)tile * WG + k) * D + 4 * lane));
            const uint32_t wk[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll 4
            for (int j = 0; j < E; ++j) {
                const int i = k * E + j;
                if (i >= ntok) break;
                __half o[4];
                if (all_exact) {
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        o[c] = __float2half_rn(fmaf((float)((wk[c] >> (j * BITS)) & MASK), s[c], z[c]));
                } else {
#pragma unroll
                    for (int c = 0; c < 4; ++c) o[c] = recon_exact((wk[c] >> (j * BITS)) & MASK, s[c], z[c]);
                }
                const __half2 a = __halves2half2(o[0], o[1]), b = __halves2half2(o[2], o[3]);
                *reinterpret_cast<uint2 *>(static_cast<__half *>(p.out) + ((size_t)bh * p.S_q + g * G + i) * D + 4 * lane) =
                    make_uint2(*reinterpret_cast<const uint32_t *>(&a), *reinterpret_cast<const uint32_t *>(&b));
            }
        }
    }
}

// ------------------------------------------------------------ launchers

template <int BITS, int G>
cudaError_t launch_q(const KiviQuantParams &p, bool per_channel, cudaStream_t stream)
{
    const int sms = sm_count();
    if (per_channel) {
        auto kern = kivi_keys_kernel<BITS, G>;
        constexpr int smem = key_smem<G>();
        constexpr int warps = key_warps<G>();
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        const int ntiles = p.B * p.H * ((p.S_q + G - 1) / G);
        int grid = (ntiles + warps - 1) / warps;
        if (grid > sms) grid = sms;
        if (grid < 1) grid = 1;
        kern<<<grid, warps * 32, smem, stream>>>(p);
    } else {
        auto kern = kivi_values_kernel<BITS, G>;
        constexpr int smem = val_smem(BITS, G);
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        const int nblk = (p.B * p.H * p.S_q + 31) / 32;
        int grid = (nblk + VAL_WARPS - 1) / VAL_WARPS;
        if (grid > sms) grid = sms;
        if (grid < 1) grid = 1;
        kern<<<grid, VAL_WARPS * 32, smem, stream>>>(p);
    }
    return cudaGetLastError();
}

template <int BITS, int G>
cudaError_t launch_dq(const KiviDequantParams &p, bool per_channel, cudaStream_t stream)
{
    const int cap = sm_count() * 8;
    if (per_channel) {
        const int ntiles = p.BH * p.NG;
        int grid = (ntiles + DQ_THREADS / 32 - 1) / (DQ_THREADS / 32);
        if (grid > cap) grid = cap;
        if (grid < 1) grid = 1;
        kivi_keys_dequant_kernel<BITS, G><<<grid, DQ_THREADS, 0, stream>>>(p);
    } else {
        auto kern = kivi_values_dequant_kernel<BITS, G>;
        constexpr int smem = vdq_smem(BITS);
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        const int nblk = (p.BH * p.S_q + 31) / 32;
        int grid = (nblk + VDQ_WARPS - 1) / VDQ_WARPS;
        if (grid > sm_count()) grid = sm_count();
        if (grid < 1) grid = 1;
        kern<<<grid, VDQ_WARPS * 32, smem, stream>>>(p);
    }
    return cudaGetLastError();
}

template <int BITS>
cudaError_t dispatch_q(const KiviQuantParams &p, bool per_channel, cudaStream_t stream)
{
    switch (p.group) {
    case 32: return launch_q<BITS, 32>(p, per_channel, stream);
    case 64: return launch_q<BITS, 64>(p, per_channel, stream);
    case 128: return launch_q<BITS, 128>(p, per_channel, stream);
    default: return cudaErrorInvalidValue;
    }
}

template <int BITS>
cudaError_t dispatch_dq(const KiviDequantParams &p, bool per_channel, cudaStream_t stream)
{
    switch (p.group) {
    case 32: return launch_dq<BITS, 32>(p, per_channel, stream);
    case 64: return launch_dq<BITS, 64>(p, per_channel, stream);
    case 128: return launch_dq<BITS, 128>(p, per_channel, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_kivi_quant(const KiviQuantParams &p, int bits, bool per_channel, cudaStream_t stream)
{
    if (p.B * p.H <= 0 || p.S_q <= 0) return cudaSuccess;
    switch (bits) {
    case 1: return dispatch_q<1>(p, per_channel, stream);
    case 2: return dispatch_q<2>(p, per_channel, stream);
    case 4: return dispatch_q<4>(p, per_channel, stream);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_kivi_dequant(const KiviDequantParams &p, int bits, bool per_channel, cudaStream_t stream)
{
    if (p.BH <= 0 || p.S_q <= 0) return cudaSuccess;
    switch (bits) {
    case 1: return dispatch_dq<1>(p, per_channel, stream);
    case 2: return dispatch_dq<2>(p, per_channel, stream);
    case 4: return dispatch_dq<4>(p, per_channel, stream);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t kivi_take_device_error(unsigned *bits, cudaStream_t stream)
{
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(bits, g_kivi_err, sizeof(unsigned), 0,
                                              cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    if (*bits) e = cudaMemcpyToSymbolAsync(g_kivi_err, &zero, sizeof(unsigned), 0,
                                           cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return e;
    return cudaStreamSynchronize(stream);
}

}  // namespace vq
