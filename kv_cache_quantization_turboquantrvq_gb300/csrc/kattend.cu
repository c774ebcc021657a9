// kattend.cu - decode-time attention over a KIVI cache with the dequantization
// inside the attention (sm_103a).
//
// Method (VeloxQuant-MLX blog, tag "kivi": the first post's closing section,
// "Dequant-in-SDPA - teach attention to read packed codes directly, so
// expansion happens in registers and never in RAM"; the reconstruction is the
// quantizer's g_hat = q * scale + zero, second post, "What KIVI is").  Keys
// are quantized per channel over groups of G tokens, values per token over
// groups of G channels (the flush kernels' layouts); the last R tokens of a
// sequence are the fp16 residual window.
//
// Keys.  With the group's scale s and zero z of channel d,
//   q . k_t = sum_d (q_d s_d) code_{t,d} + sum_d q_d z_d,
// so a 32-token tile (inside one key group: G is a multiple of 32) costs one
// product q_d s_d per channel and one fused multiply-add per code.  Key words
// are channel-major (one word holds consecutive tokens of a channel), so lane
// (tg, cg) = (lane >> 3, lane & 7) takes tokens 8 tg .. 8 tg + 7 and channels
// 16 cg .. 16 cg + 15: its partial dot products are reduced over the 8 lanes
// of its token group by an exchange that leaves token `lane` on lane `lane`
// (one key per lane for the online softmax).  Codes become floats by the
// 2^23 magic-number trick (OR into the mantissa of 2^23, subtract 2^23), two
// tokens at a time, so the arithmetic runs as paired FMAs.
// Values.  sum_t w_t (code_{t,d} s_t + z_t) = sum_t (w_t s_t) code_{t,d} +
// sum_t w_t z_t: lanes own 4 coordinates (inside one value group), two tokens
// per paired FMA.
// Grid, staging and merging as the RVQ attention: fixed-size chunks of the
// quantized tokens per CTA, one more CTA per (sequence, kv head) for the
// residual window, per-warp double-buffered bulk copies (key words, the
// group's key scale and zero, value words, value scales and zeros), partials
// (max, sum, unnormalised output) merged by a combine kernel.
#include <cuda_fp16.h>

#include "device_common.cuh"
#include "launch.h"

namespace vq {

namespace {

VQ_DEFINE_ERROR_WORD(g_ka_err);

constexpr int D = 128;
constexpr int KA_WARPS = 8;
constexpr int KT = 32;  // tokens per warp tile
constexpr int KA_STAGES = 2;
constexpr float NEG_INF = -__builtin_huge_valf();
constexpr float TWO23 = 8388608.0f;

__host__ __device__ constexpr int ka_stage(int bits, int G)
{
    // key words (bits rows of 128), key scale + zero (2 x 256 B), value words
    // (32 rows of 4 bits words), value scales + zeros (2 x 32 x 128/G halves)
    return bits * 512 + 512 + KT * 16 * bits + 2 * KT * (D / G) * 2;
}
// The stage area also serves the final merge of the warps (m, l and the
// unnormalised outputs of every warp), so it is at least that large.
__host__ __device__ constexpr int ka_region(int bits, int G, int GQ)
{
    return KA_WARPS * KA_STAGES * ka_stage(bits, G) > KA_WARPS * GQ * (D + 2) * 4
               ? KA_WARPS * KA_STAGES * ka_stage(bits, G)
               : KA_WARPS * GQ * (D + 2) * 4;
}
__host__ __device__ constexpr int ka_smem(int bits, int G, int GQ)
{
    // query [g][d], weights [warp][token][g], stages / merge, mbarriers
    return D * GQ * 4 + KA_WARPS * KT * GQ * 4 + ka_region(bits, G, GQ) + KA_WARPS * KA_STAGES * 8;
}

__device__ __forceinline__ int ord_of(float x)
{
    const int i = __float_as_int(x);
    return i >= 0 ? i : i ^ 0x7fffffff;
}
__device__ __forceinline__ float float_of_ord(int i) { return __int_as_float(i >= 0 ? i : i ^ 0x7fffffff); }
__device__ __forceinline__ float2 f2(float a, float b) { return make_float2(a, b); }

// 2^23 + (x & m) as a float: the code in the low mantissa bits of 2^23.
__device__ __forceinline__ float magic_code(uint32_t x, uint32_t m)
{
    return __uint_as_float((x & m) | 0x4B000000u);
}

// Load and scale the GQ query rows of kv head h (fp32, times scale * log2 e).
template <int GQ>
__device__ __forceinline__ void ka_load_query(const KiviAttendParams &p, int b, int h, float *qf)
{
    for (int i = threadIdx.x; i < GQ * D; i += blockDim.x) {
        const int g = i / D, d = i - g * D;
        const __half v = static_cast<const __half *>(p.q)[((size_t)b * p.Hq + (size_t)h * GQ + g) * D + d];
        qf[g * D + d] = __half2float(v) * p.qscale;
    }
}

// Merge the warps' (m, l, o) through shared memory and write the output (one
// part) or this part's partial.  o holds the lane's coordinates cbase .. + 3
// (the 32 lanes of a warp cover all 128).
template <int GQ>
__device__ __forceinline__ void ka_merge_write(const KiviAttendParams &p, unsigned char *scratch, int b, int h,
                                               int part, int nparts, const float (&m)[GQ], const float (&l)[GQ],
                                               const float (&o)[GQ][4], int cbase)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nw = blockDim.x >> 5;
    float *ms = reinterpret_cast<float *>(scratch);
    float *ls = ms + nw * GQ;
    float *os = ls + nw * GQ;
#pragma unroll
    for (int g = 0; g < GQ; ++g) {
        if (lane == 0) {
            ms[warp * GQ + g] = m[g];
            ls[warp * GQ + g] = l[g];
        }
        *reinterpret_cast<float4 *>(os + (warp * GQ + g) * D + cbase) = make_float4(o[g][0], o[g][1], o[g][2], o[g][3]);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < GQ * D; i += blockDim.x) {
        const int g = i / D, d = i - g * D;
        float M = NEG_INF;
        for (int k = 0; k < nw; ++k) M = fmaxf(M, ms[k * GQ + g]);
        float Ls = 0.0f, O = 0.0f;
        for (int k = 0; k < nw; ++k) {
            const float mk = ms[k * GQ + g];
            const float f = (mk == NEG_INF) ? 0.0f : exp2f(mk - M);
            Ls = fmaf(ls[k * GQ + g], f, Ls);
            O = fmaf(os[(k * GQ + g) * D + d], f, O);
        }
        const int hq = h * GQ + g;
        if (nparts == 1) {
            static_cast<__half *>(p.out)[((size_t)b * p.Hq + hq) * D + d] = __float2half_rn(Ls > 0.0f ? O / Ls : 0.0f);
        } else {
            float *wp = p.ws + (((size_t)b * p.Hq + hq) * nparts + part) * AT_PART;
            if (d == 0) {
                wp[0] = M;
                wp[1] = Ls;
            }
            wp[2 + d] = O;
        }
    }
}

// One chunk of the quantized tokens of one (sequence, kv head).
template <int BITS, int G, int GQ>
__global__ void __launch_bounds__(KA_WARPS * 32, 1) kivi_attend_kernel(const __grid_constant__ KiviAttendParams p)
{
    constexpr int STG = ka_stage(BITS, G);
    constexpr int KW = BITS * 512;            // key words of a tile (bytes)
    constexpr int VW = KT * 16 * BITS;        // value words of a tile (bytes)
    constexpr int VS = KT * (D / G) * 2;      // value scales (or zeros) of a tile (bytes)
    constexpr int W = D * BITS / 32;          // value words per token
    constexpr uint32_t MASK = (1u << BITS) - 1u;
    extern __shared__ __align__(128) unsigned char smem[];
    float *qf = reinterpret_cast<float *>(smem);
    float *wb = qf + GQ * D;
    unsigned char *stages = reinterpret_cast<unsigned char *>(wb + KA_WARPS * KT * GQ);
    uint64_t *bars = reinterpret_cast<uint64_t *>(stages + ka_region(BITS, G, GQ));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.y, split = blockIdx.x;
    const int b = bh / p.Hkv, h = bh - b * p.Hkv;
    int len = p.lens ? __ldg(p.lens + b) : p.S_cap;
    len = len < 0 ? 0 : (len > p.S_cap ? p.S_cap : len);
    const int s0 = split * p.chunk;
    const int nparts = p.nsplit + (p.R > 0 ? 1 : 0);
    if (s0 >= len && nparts > 1) return;  // nothing here: the combine skips this part
    const int s1 = min(len, s0 + p.chunk);
    const int ntiles = s1 > s0 ? (s1 - s0 + KT - 1) / KT : 0;

    unsigned char *my_st = stages + warp * KA_STAGES * STG;
    uint64_t *my_bar = bars + warp * KA_STAGES;
    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < KA_STAGES; ++s) mbar_init(&my_bar[s], 1);
        fence_mbar_init();
    }
    __syncwarp();
    const uint64_t pol = l2_policy_evict_first();
    const size_t tbase = (size_t)bh * p.S_cap;  // token rows of this (b, h)
    auto issue = [&](int t, int st) {
        if (lane == 0) {
            const int t0 = s0 + t * KT;
            const int g = t0 / G;
            const int w0 = (t0 % G) * BITS / 32;
            const size_t gi = (size_t)bh * p.NG + g;
            unsigned char *dst = my_st + st * STG;
            mbar_arrive_expect_tx(&my_bar[st], (uint32_t)STG);
            bulk_g2s(dst, p.kp + (gi * (G * BITS / 32) + w0) * D, KW, &my_bar[st], pol);
            bulk_g2s(dst + KW, static_cast<const __half *>(p.ks) + gi * D, 256, &my_bar[st], pol);
            bulk_g2s(dst + KW + 256, static_cast<const __half *>(p.kz) + gi * D, 256, &my_bar[st], pol);
            bulk_g2s(dst + KW + 512, p.vp + (tbase + t0) * W, VW, &my_bar[st], pol);
            bulk_g2s(dst + KW + 512 + VW, static_cast<const __half *>(p.vs) + (tbase + t0) * (D / G), VS, &my_bar[st], pol);
            bulk_g2s(dst + KW + 512 + VW + VS, static_cast<const __half *>(p.vz) + (tbase + t0) * (D / G), VS,
                     &my_bar[st], pol);
        }
    };
#pragma unroll
    for (int s = 0; s < KA_STAGES; ++s) {
        const int t = warp + s * KA_WARPS;
        if (t < ntiles) issue(t, s);
    }
    ka_load_query<GQ>(p, b, h, qf);
    __syncthreads();

    const int tg = lane >> 3, cg = lane & 7;
    // key bits of this lane's 8 tokens: word kw0, from bit ksh; token j's code
    // sits at bit j * BITS of x = word >> ksh (b = 4: tokens 4..7 at bit
    // 4 (j - 4) of x >> 16, so that every masked code stays below 2^20)
    constexpr int KBITS8 = 8 * BITS;
    const int kw0 = (tg * KBITS8) / 32, ksh = (tg * KBITS8) % 32;
    // values: lane (vh, cl) takes coordinates 8 cl .. 8 cl + 7 (one value
    // group) of the tokens of parity vh; their codes at bit c * BITS of
    // word vwi >> vsh (b = 4: coordinates 4..7 of the high half)
    const int vh = lane >> 4, cl = lane & 15;
    const int vwi = (8 * cl * BITS) / 32, vsh = (8 * cl * BITS) % 32, vj = (8 * cl) / G;
    float *my_w = wb + warp * KT * GQ;

    float m[GQ], l[GQ], zb[GQ];
    float2 o2[GQ][4];  // coordinate pairs (2i, 2i + 1) of the lane's 8, scaled by 2^(code shift)
#pragma unroll
    for (int g = 0; g < GQ; ++g) {
        m[g] = NEG_INF;
        l[g] = 0.0f;
        zb[g] = 0.0f;  // sum of w z (the value zeros' share), per head
#pragma unroll
        for (int i = 0; i < 4; ++i) o2[g][i] = f2(0.0f, 0.0f);
    }

    for (int it = 0;; ++it) {
        const int t = warp + it * KA_WARPS;
        if (t >= ntiles) break;
        const int st = it % KA_STAGES;
        const int t0 = s0 + t * KT;
        const int n = min(KT, s1 - t0);
        const bool ok = mbar_wait_bounded(&my_bar[st], (uint32_t)(it / KA_STAGES) & 1u);
        if (!__all_sync(FULL_MASK, ok)) {
            if (lane == 0) atomicOr(&g_ka_err, (unsigned)VQ_DEVERR_WAIT_TIMEOUT);
            for (int k = 1; k < KA_STAGES; ++k) {
                const int it2 = it + k;
                if (warp + it2 * KA_WARPS < ntiles)
                    (void)mbar_wait_bounded(&my_bar[it2 % KA_STAGES], (uint32_t)(it2 / KA_STAGES) & 1u);
            }
            break;
        }
        const unsigned char *sb = my_st + st * STG;
        const uint32_t *kwords = reinterpret_cast<const uint32_t *>(sb) + kw0 * D;
        const __half *ksc = reinterpret_cast<const __half *>(sb + KW);
        const __half *kze = reinterpret_cast<const __half *>(sb + KW + 256);

        // ---- scores: partial dot products over this lane's 16 channels for
        // its 8 tokens (token pairs in the two halves of a float2), each code
        // scaled by 2^(its bit offset) until the end of the channel loop
        float2 acc[4][GQ];
        float bias[GQ];
#pragma unroll
        for (int g = 0; g < GQ; ++g) {
            bias[g] = 0.0f;
#pragma unroll
            for (int jp = 0; jp < 4; ++jp) acc[jp][g] = f2(0.0f, 0.0f);
        }
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
            const int d0 = cg * 16 + c4 * 4;
            const uint4 wv = *reinterpret_cast<const uint4 *>(kwords + d0);
            const uint2 sv = *reinterpret_cast<const uint2 *>(ksc + d0);
            const uint2 zv = *reinterpret_cast<const uint2 *>(kze + d0);
            const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
            const float2 s01 = __half22float2(*reinterpret_cast<const __half2 *>(&sv.x));
            const float2 s23 = __half22float2(*reinterpret_cast<const __half2 *>(&sv.y));
            const float2 z01 = __half22float2(*reinterpret_cast<const __half2 *>(&zv.x));
            const float2 z23 = __half22float2(*reinterpret_cast<const __half2 *>(&zv.y));
            const float sc[4] = {s01.x, s01.y, s23.x, s23.y};
            const float ze[4] = {z01.x, z01.y, z23.x, z23.y};
            float qd[GQ][4];
#pragma unroll
            for (int g = 0; g < GQ; ++g) {
                const float4 q4 = *reinterpret_cast<const float4 *>(qf + g * D + d0);
                qd[g][0] = q4.x; qd[g][1] = q4.y; qd[g][2] = q4.z; qd[g][3] = q4.w;
            }
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint32_t x = ww[c] >> ksh;
                const uint32_t xh = BITS == 4 ? x >> 16 : x;
                float2 cf[4];
#pragma unroll
                for (int jp = 0; jp < 4; ++jp) {
                    const int j0 = 2 * jp, j1 = 2 * jp + 1;
                    const uint32_t s0b = (uint32_t)((BITS == 4 && j0 >= 4 ? j0 - 4 : j0) * BITS);
                    const uint32_t s1b = (uint32_t)((BITS == 4 && j1 >= 4 ? j1 - 4 : j1) * BITS);
                    const uint32_t src0 = (BITS == 4 && j0 >= 4) ? xh : x;
                    const uint32_t src1 = (BITS == 4 && j1 >= 4) ? xh : x;
                    cf[jp] = __fadd2_rn(f2(magic_code(src0, MASK << s0b), magic_code(src1, MASK << s1b)),
                                        f2(-TWO23, -TWO23));
                }
#pragma unroll
                for (int g = 0; g < GQ; ++g) {
                    const float qk = qd[g][c] * sc[c];
                    bias[g] = fmaf(qd[g][c], ze[c], bias[g]);
#pragma unroll
                    for (int jp = 0; jp < 4; ++jp) acc[jp][g] = __ffma2_rn(f2(qk, qk), cf[jp], acc[jp][g]);
                }
            }
        }
        // undo the code scales (exact powers of two) and add the zero term
        float v8[8][GQ];
#pragma unroll
        for (int jp = 0; jp < 4; ++jp) {
            const int j0 = 2 * jp, j1 = 2 * jp + 1;
            const float u0 = __int_as_float((127 - (BITS == 4 && j0 >= 4 ? j0 - 4 : j0) * BITS) << 23);
            const float u1 = __int_as_float((127 - (BITS == 4 && j1 >= 4 ? j1 - 4 : j1) * BITS) << 23);
#pragma unroll
            for (int g = 0; g < GQ; ++g) {
                v8[j0][g] = fmaf(acc[jp][g].x, u0, bias[g]);
                v8[j1][g] = fmaf(acc[jp][g].y, u1, bias[g]);
            }
        }
        // ---- reduce over the 8 lanes of the token group: exchange on the
        // token bits so that lane cg ends with token cg (all heads)
        {
            const bool hi4 = (cg & 4) != 0;
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int g = 0; g < GQ; ++g) {
                    const float keep = hi4 ? v8[4 + i][g] : v8[i][g];
                    const float send = hi4 ? v8[i][g] : v8[4 + i][g];
                    v8[i][g] = keep + __shfl_xor_sync(FULL_MASK, send, 4);
                }
            const bool hi2 = (cg & 2) != 0;
#pragma unroll
            for (int i = 0; i < 2; ++i)
#pragma unroll
                for (int g = 0; g < GQ; ++g) {
                    const float keep = hi2 ? v8[2 + i][g] : v8[i][g];
                    const float send = hi2 ? v8[i][g] : v8[2 + i][g];
                    v8[i][g] = keep + __shfl_xor_sync(FULL_MASK, send, 2);
                }
            const bool hi1 = (cg & 1) != 0;
#pragma unroll
            for (int g = 0; g < GQ; ++g) {
                const float keep = hi1 ? v8[1][g] : v8[0][g];
                const float send = hi1 ? v8[0][g] : v8[1][g];
                v8[0][g] = keep + __shfl_xor_sync(FULL_MASK, send, 1);
            }
        }

        // ---- online softmax over the tile (token `lane` on this lane)
        const bool valid = lane < n;
        float wv[GQ];
#pragma unroll
        for (int g = 0; g < GQ; ++g) {
            const float sc = valid ? v8[0][g] : NEG_INF;
            const float mt = float_of_ord(__reduce_max_sync(FULL_MASK, ord_of(sc)));
            if (mt > m[g]) {  // warp-uniform
                const float f = exp2f(m[g] - mt);
                l[g] *= f;
                zb[g] *= f;
#pragma unroll
                for (int i = 0; i < 4; ++i) o2[g][i] = __fmul2_rn(o2[g][i], f2(f, f));
                m[g] = mt;
            }
            wv[g] = exp2f(sc - m[g]);
            l[g] += wv[g];
        }
#pragma unroll
        for (int g = 0; g < GQ; ++g) my_w[lane * GQ + g] = wv[g];
        __syncwarp();

        // ---- values: lane (vh, cl), coordinates 8 cl .. 8 cl + 7 of the
        // tokens k = vh, vh + 2, ...; coordinate pairs per paired FMA
        {
            const uint32_t *vwords = reinterpret_cast<const uint32_t *>(sb + KW + 512);
            const __half *vsc = reinterpret_cast<const __half *>(sb + KW + 512 + VW);
            const __half *vze = reinterpret_cast<const __half *>(sb + KW + 512 + VW + VS);
            auto token = [&](int k) {
                const uint32_t x = vwords[k * W + vwi] >> vsh;
                const uint32_t xh = BITS == 4 ? x >> 16 : x;
                const float sk = __half2float(vsc[k * (D / G) + vj]);
                const float zk = __half2float(vze[k * (D / G) + vj]);
                float2 cf[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int c0 = 2 * i, c1 = 2 * i + 1;
                    const uint32_t s0b = (uint32_t)((BITS == 4 && c0 >= 4 ? c0 - 4 : c0) * BITS);
                    const uint32_t s1b = (uint32_t)((BITS == 4 && c1 >= 4 ? c1 - 4 : c1) * BITS);
                    const uint32_t src0 = (BITS == 4 && c0 >= 4) ? xh : x;
                    const uint32_t src1 = (BITS == 4 && c1 >= 4) ? xh : x;
                    cf[i] = __fadd2_rn(f2(magic_code(src0, MASK << s0b), magic_code(src1, MASK << s1b)),
                                       f2(-TWO23, -TWO23));
                }
                float wk[GQ];
                if constexpr (GQ == 1) {
                    wk[0] = my_w[k];
                } else if constexpr (GQ == 2) {
                    const float2 w2 = *reinterpret_cast<const float2 *>(my_w + k * 2);
                    wk[0] = w2.x; wk[1] = w2.y;
                } else {
#pragma unroll
                    for (int g = 0; g < GQ; g += 4) {
                        const float4 w4 = *reinterpret_cast<const float4 *>(my_w + k * GQ + g);
                        wk[g] = w4.x; wk[g + 1] = w4.y; wk[g + 2] = w4.z; wk[g + 3] = w4.w;
                    }
                }
#pragma unroll
                for (int g = 0; g < GQ; ++g) {
                    const float a = wk[g] * sk;
                    zb[g] = fmaf(wk[g], zk, zb[g]);
#pragma unroll
                    for (int i = 0; i < 4; ++i) o2[g][i] = __ffma2_rn(f2(a, a), cf[i], o2[g][i]);
                }
            };
            if (n == KT) {
#pragma unroll 4
                for (int k = vh; k < KT; k += 2) token(k);
            } else {
                for (int k = vh; k < n; k += 2) token(k);
            }
        }

        __syncwarp();
        fence_proxy_async_smem();
        if (t + KA_STAGES * KA_WARPS < ntiles) issue(t + KA_STAGES * KA_WARPS, st);
    }

    // l: each lane summed its own tokens' weights; the value halves (vh = 0, 1)
    // hold the even and odd tokens of the same 8 coordinates: add them, undo
    // the code scales, and fold in the zeros' share (one value group per lane)
    float o[GQ][4];
#pragma unroll
    for (int g = 0; g < GQ; ++g) {
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) l[g] += __shfl_xor_sync(FULL_MASK, l[g], off);
        zb[g] += __shfl_xor_sync(FULL_MASK, zb[g], 16);
        float full[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float ox = o2[g][i].x + __shfl_xor_sync(FULL_MASK, o2[g][i].x, 16);
            const float oy = o2[g][i].y + __shfl_xor_sync(FULL_MASK, o2[g][i].y, 16);
            const int c0 = 2 * i, c1 = 2 * i + 1;
            const float u0 = __int_as_float((127 - (BITS == 4 && c0 >= 4 ? c0 - 4 : c0) * BITS) << 23);
            const float u1 = __int_as_float((127 - (BITS == 4 && c1 >= 4 ? c1 - 4 : c1) * BITS) << 23);
            full[c0] = fmaf(ox, u0, zb[g]);
            full[c1] = fmaf(oy, u1, zb[g]);
        }
        // this lane publishes coordinates 8 cl + 4 vh .. + 3
#pragma unroll
        for (int c = 0; c < 4; ++c) o[g][c] = vh ? full[4 + c] : full[c];
    }
    __syncthreads();
    ka_merge_write<GQ>(p, stages, b, h, split, nparts, m, l, o, 8 * cl + 4 * vh);
}

// The fp16 residual window of one (sequence, kv head): warp w takes tokens
// w, w + 8, ...; lanes own 4 channels for the dot product (warp sum) and 4
// coordinates for the values.  Writes part nsplit.
template <int GQ>
__global__ void __launch_bounds__(KA_WARPS * 32) kivi_attend_residual_kernel(const __grid_constant__ KiviAttendParams p)
{
    __shared__ float qf[GQ * D];
    __shared__ __align__(16) unsigned char scratch[KA_WARPS * GQ * (D + 2) * 4];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.x;
    const int b = bh / p.Hkv, h = bh - b * p.Hkv;
    int rl = p.res_lens ? __ldg(p.res_lens + b) : p.R;
    rl = rl < 0 ? 0 : (rl > p.R ? p.R : rl);
    const int nparts = p.nsplit + 1;
    if (rl == 0) return;  // the combine skips an empty window
    ka_load_query<GQ>(p, b, h, qf);
    __syncthreads();
    float qv[GQ][4];
#pragma unroll
    for (int g = 0; g < GQ; ++g)
#pragma unroll
        for (int c = 0; c < 4; ++c) qv[g][c] = qf[g * D + 4 * lane + c];
    float m[GQ], l[GQ], o[GQ][4];
#pragma unroll
    for (int g = 0; g < GQ; ++g) {
        m[g] = NEG_INF;
        l[g] = 0.0f;
#pragma unroll
        for (int c = 0; c < 4; ++c) o[g][c] = 0.0f;
    }
    const __half *kr = static_cast<const __half *>(p.kr) + (size_t)bh * p.R * D;
    const __half *vr = static_cast<const __half *>(p.vr) + (size_t)bh * p.R * D;
    for (int r = warp; r < rl; r += KA_WARPS) {
        const uint2 ku = __ldg(reinterpret_cast<const uint2 *>(kr + (size_t)r * D) + lane);
        const uint2 vu = __ldg(reinterpret_cast<const uint2 *>(vr + (size_t)r * D) + lane);
        const float2 k01 = __half22float2(*reinterpret_cast<const __half2 *>(&ku.x));
        const float2 k23 = __half22float2(*reinterpret_cast<const __half2 *>(&ku.y));
        const float2 v01 = __half22float2(*reinterpret_cast<const __half2 *>(&vu.x));
        const float2 v23 = __half22float2(*reinterpret_cast<const __half2 *>(&vu.y));
        const float kk[4] = {k01.x, k01.y, k23.x, k23.y};
        const float vv[4] = {v01.x, v01.y, v23.x, v23.y};
#pragma unroll
        for (int g = 0; g < GQ; ++g) {
            float s = 0.0f;
#pragma unroll
            for (int c = 0; c < 4; ++c) s = fmaf(qv[g][c], kk[c], s);
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) s += __shfl_xor_sync(FULL_MASK, s, off);
            const float mn = fmaxf(m[g], s);
            const float f = exp2f(m[g] - mn);
            const float w = exp2f(s - mn);
            l[g] = l[g] * f + w;
#pragma unroll
            for (int c = 0; c < 4; ++c) o[g][c] = fmaf(w, vv[c], o[g][c] * f);
            m[g] = mn;
        }
    }
    // l is already the warp's total (every lane holds the same sums)
    ka_merge_write<GQ>(p, scratch, b, h, p.nsplit, nparts, m, l, o, 4 * lane);
}

// Combine the parts of one (sequence, query head): the quantized chunks that
// hold tokens and the residual window when it holds any.
__global__ void __launch_bounds__(D) kivi_attend_combine_kernel(const __grid_constant__ KiviAttendParams p)
{
    const int bq = blockIdx.x, d = threadIdx.x;
    const int b = bq / p.Hq;
    int len = p.lens ? __ldg(p.lens + b) : p.S_cap;
    len = len < 0 ? 0 : (len > p.S_cap ? p.S_cap : len);
    int rl = p.res_lens ? __ldg(p.res_lens + b) : p.R;
    rl = rl < 0 ? 0 : (rl > p.R ? p.R : rl);
    const int nparts = p.nsplit + (p.R > 0 ? 1 : 0);
    const int nv = (len + p.chunk - 1) / p.chunk;
    const float *wp = p.ws + (size_t)bq * nparts * AT_PART;
    float M = NEG_INF;
    for (int s = 0; s < nv; ++s) M = fmaxf(M, wp[(size_t)s * AT_PART]);
    if (rl > 0) M = fmaxf(M, wp[(size_t)p.nsplit * AT_PART]);
    float Ls = 0.0f, O = 0.0f;
    for (int s = 0; s < nv; ++s) {
        const float ms = wp[(size_t)s * AT_PART];
        const float f = (ms == NEG_INF) ? 0.0f : exp2f(ms - M);
        Ls = fmaf(wp[(size_t)s * AT_PART + 1], f, Ls);
        O = fmaf(wp[(size_t)s * AT_PART + 2 + d], f, O);
    }
    if (rl > 0) {
        const float *r = wp + (size_t)p.nsplit * AT_PART;
        const float f = (r[0] == NEG_INF) ? 0.0f : exp2f(r[0] - M);
        Ls = fmaf(r[1], f, Ls);
        O = fmaf(r[2 + d], f, O);
    }
    static_cast<__half *>(p.out)[(size_t)bq * D + d] = __float2half_rn(Ls > 0.0f ? O / Ls : 0.0f);
}

template <int BITS, int G, int GQ>
cudaError_t launch_ka(const KiviAttendParams &p, cudaStream_t stream)
{
    auto kern = kivi_attend_kernel<BITS, G, GQ>;
    constexpr int smem = ka_smem(BITS, G, GQ);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int nparts = p.nsplit + (p.R > 0 ? 1 : 0);
    dim3 grid(p.nsplit, p.B * p.Hkv);
    kern<<<grid, KA_WARPS * 32, smem, stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (p.R > 0) {
        kivi_attend_residual_kernel<GQ><<<p.B * p.Hkv, KA_WARPS * 32, 0, stream>>>(p);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (nparts == 1) return cudaSuccess;
    kivi_attend_combine_kernel<<<p.B * p.Hq, D, 0, stream>>>(p);
    return cudaGetLastError();
}

template <int BITS, int G>
cudaError_t dispatch_ka_gq(const KiviAttendParams &p, cudaStream_t stream)
{
    switch (p.Hq / p.Hkv) {
    case 1: return launch_ka<BITS, G, 1>(p, stream);
    case 2: return launch_ka<BITS, G, 2>(p, stream);
    case 4: return launch_ka<BITS, G, 4>(p, stream);
    case 8: return launch_ka<BITS, G, 8>(p, stream);
    default: return cudaErrorInvalidValue;
    }
}

template <int BITS>
cudaError_t dispatch_ka_g(const KiviAttendParams &p, cudaStream_t stream)
{
    switch (p.G) {
    case 32: return dispatch_ka_gq<BITS, 32>(p, stream);
    case 64: return dispatch_ka_gq<BITS, 64>(p, stream);
    case 128: return dispatch_ka_gq<BITS, 128>(p, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_kivi_attend(const KiviAttendParams &p, int bits, cudaStream_t stream)
{
    if (p.B <= 0 || p.Hq <= 0) return cudaSuccess;
    switch (bits) {
    case 1: return dispatch_ka_g<1>(p, stream);
    case 2: return dispatch_ka_g<2>(p, stream);
    case 4: return dispatch_ka_g<4>(p, stream);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t kivi_attend_take_device_error(unsigned *bits, cudaStream_t stream)
{
    *bits = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(bits, g_ka_err, sizeof(unsigned), 0, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    if (*bits) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbolAsync(g_ka_err, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice, stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    }
    return e;
}

}  // namespace vq
