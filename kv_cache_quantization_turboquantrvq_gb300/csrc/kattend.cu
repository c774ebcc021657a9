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
// a dense product of the tile's codes [32 tokens x 128 channels] with the
// columns (q s) of the GQ query heads.  Values, with the token's scale s_t and
// zero z_t of the coordinate's group,
//   sum_t w_t v_{t,d} = sum_t code_{t,d} (w_t s_t) + sum_t w_t z_t,
// a dense product of the codes [128 coordinates x 32 tokens] with the columns
// (w s).  Both run on the tensor cores as 16 x 8 x 16 tiles (mma.sync, fp16
// operands, fp32 accumulation): the codes are exact in fp16 (byte-permuted
// into place, masked into the mantissa of 1024 and 1024 subtracted, each row
// still scaled by a power of two that the epilogue removes), and every float
// column is carried as two fp16 columns, u rounded to fp16 and the rounded
// rest, so a head's products keep about 22 bits.  The 8 columns of a tile are
// 4 heads x (hi, lo).  The tensor-core rate is not the limit (the columns are
// few): the gain is that one instruction does 2048 multiply-adds, leaving
// the byte shuffling of the codes as the main cost.  The query
// is scaled by a power of two so that |q| <= 1 and every q s fits in fp16.
// The zero terms are plain sums (one per head and group).
// Grid, staging and merging as the RVQ attention: fixed-size chunks of the
// quantized tokens per CTA, plus one CTA per (sequence, kv head) in the same
// grid for the residual window (so it overlaps the chunks), per-warp rings of
// bulk copies (key words, the group's key scale and zero, value words, value
// scales and zeros), partials (max, sum, unnormalised output) merged by a
// combine kernel.
#include <cuda_fp16.h>

#include "device_common.cuh"
#include "launch.h"

namespace vq {

namespace {

VQ_DEFINE_ERROR_WORD(g_ka_err);

constexpr int D = 128;
constexpr int KA_WARPS = 8;
constexpr int KT = 32;  // tokens per warp tile
constexpr float NEG_INF = -__builtin_huge_valf();

__host__ __device__ constexpr int ka_stage(int bits, int G)
{
    // key words (bits rows of 128), key scale + zero (2 x 256 B), value words
    // (32 rows of 4 bits words), value scales + zeros (2 x 32 x 128/G halves)
    return bits * 512 + 512 + KT * 16 * bits + 2 * KT * (D / G) * 2;
}
// Tiles in flight per warp: three where that still leaves room for two CTAs
// per SM, else two.
__host__ __device__ constexpr int ka_nst(int bits, int G)
{
    return 3 * KA_WARPS * ka_stage(bits, G) <= 100 * 1024 ? 3 : 2;
}
// The stage area also serves the final merge of the warps (m, l and the
// unnormalised outputs of every warp), so it is at least that large.
__host__ __device__ constexpr int ka_region(int bits, int G, int GQ)
{
    return KA_WARPS * ka_nst(bits, G) * ka_stage(bits, G) > KA_WARPS * GQ * (D + 2) * 4
               ? KA_WARPS * ka_nst(bits, G) * ka_stage(bits, G)
               : KA_WARPS * GQ * (D + 2) * 4;
}
constexpr int QS = D + 16;  // query row stride (floats): rows of 4 heads fall on 2 bank halves
__host__ __device__ constexpr int ka_smem(int bits, int G, int GQ)
{
    // query [g][QS], weights [warp][g][slot], stages / merge, mbarriers
    return QS * GQ * 4 + KA_WARPS * KT * GQ * 4 + ka_region(bits, G, GQ) + KA_WARPS * ka_nst(bits, G) * 8;
}

// Load the GQ query rows of kv head h, times scale * log2 e, into qf (row
// stride STRIDE).  With `bounded`, the rows are also multiplied by the power
// of two 2^-e that brings max |entry| into [1/2, 1), and 2^e is returned: the
// products q_d s_d of the key scores then stay inside the fp16 range whatever
// the key scales (|s| <= 65504), as far from its subnormals as that allows,
// and the scores are multiplied back by 2^e, exactly.
template <int GQ, int STRIDE>
__device__ __forceinline__ float ka_load_query(const KiviAttendParams &p, int b, int h, float *qf, bool bounded)
{
    const __half *q = static_cast<const __half *>(p.q) + ((size_t)b * p.Hq + (size_t)h * GQ) * D;
    const float qs = p.qscale;
    if (!bounded) {
        for (int i = threadIdx.x; i < GQ * D; i += blockDim.x) {
            const int g = i / D, d = i - g * D;
            qf[g * STRIDE + d] = __half2float(q[i]) * qs;
        }
        return 1.0f;
    }
    // every warp loads the GQ rows once (GQ * D / 8 16-byte pieces; the rows
    // start 256-byte aligned), takes the maximum and writes the scaled rows
    // (the warps write the same values)
    constexpr int NP = GQ * D / 8;
    constexpr int PPL = (NP + 31) / 32;
    const int lane = threadIdx.x & 31;
    uint4 u[PPL];
    float mx = 0.0f;
#pragma unroll
    for (int k = 0; k < PPL; ++k) {
        const int i = lane + 32 * k;
        u[k] = i < NP ? reinterpret_cast<const uint4 *>(q)[i] : make_uint4(0u, 0u, 0u, 0u);
        const uint32_t w[4] = {u[k].x, u[k].y, u[k].z, u[k].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w[j]));
            mx = fmaxf(mx, fmaxf(fabsf(f.x), fabsf(f.y)));
        }
    }
    mx = __uint_as_float(__reduce_max_sync(FULL_MASK, __float_as_uint(mx))) * fabsf(qs);
    float pe = 1.0f, ps = 1.0f;
    if (mx >= 1.0e-30f && mx <= 1.0e30f) {
        const int ex = (int)((__float_as_uint(mx) >> 23) & 0xffu) - 126;  // 2^(ex-1) <= mx < 2^ex
        pe = __uint_as_float((uint32_t)(127 + ex) << 23);
        ps = __uint_as_float((uint32_t)(127 - ex) << 23);
    }
#pragma unroll
    for (int k = 0; k < PPL; ++k) {
        const int i = lane + 32 * k;
        if (i < NP) {
            const int g = (8 * i) / D, d = 8 * i - g * D;
            const uint32_t w[4] = {u[k].x, u[k].y, u[k].z, u[k].w};
            float v[8];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w[j]));
                v[2 * j] = f.x * qs * ps;
                v[2 * j + 1] = f.y * qs * ps;
            }
            *reinterpret_cast<float4 *>(qf + g * STRIDE + d) = make_float4(v[0], v[1], v[2], v[3]);
            *reinterpret_cast<float4 *>(qf + g * STRIDE + d + 4) = make_float4(v[4], v[5], v[6], v[7]);
        }
    }
    return pe;
}

// Merge the warps' (m, l, o) staged in shared memory (ms[warp][g],
// ls[warp][g], os[warp][g][d]) and write the output (one part) or this part's
// partial.
template <int GQ>
__device__ __forceinline__ void ka_merge_finish(const KiviAttendParams &p, unsigned char *scratch, int b, int h,
                                                int part, int nparts)
{
    const int nw = blockDim.x >> 5;
    const float *ms = reinterpret_cast<const float *>(scratch);
    const float *ls = ms + nw * GQ;
    const float *os = ls + nw * GQ;
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

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }
__device__ __forceinline__ __half2 bits_h2(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }

// The fp16 pair of this lane's part of u: hi lanes (mh = ~0x1fff, ml = 0)
// take u with its mantissa cut to fp16's 10 bits (exact in fp16), lo lanes
// (mh = ~0, ml = ~0x1fff) the rest u - hi, rounded to fp16: the two columns
// of one head together carry u to about 21 bits.
__device__ __forceinline__ uint32_t split_pack(float2 u, uint32_t mh, uint32_t ml)
{
    const uint32_t ux = __float_as_uint(u.x), uy = __float_as_uint(u.y);
    const float2 a = make_float2(__uint_as_float(ux & mh), __uint_as_float(uy & mh));
    const float2 c = make_float2(__uint_as_float((ux & ml) ^ 0x80000000u), __uint_as_float((uy & ml) ^ 0x80000000u));
    return h2_bits(__float22half2_rn(__fadd2_rn(a, c)));
}

// code * 2^shift in each half of x's masked bits: OR-ing them into the
// mantissa of 1024 and subtracting 1024 is exact.  (Codes left as fp16
// subnormals, with no subtraction, lose precision in the tile products.)
__device__ __forceinline__ uint32_t code_h2(uint32_t x, uint32_t m)
{
    return h2_bits(__hsub2(bits_h2((x & m) | 0x64006400u), bits_h2(0x64006400u)));
}

// d += a * b for one 16 x 8 x 16 tile, fp16 operands, fp32 accumulation.
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t quad_at(const uint4 &v, int i)
{
    return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

// Up to 4 fp16 scales (or zeros) of one token's value groups, as floats.
template <int NV>
__device__ __forceinline__ void load_groups(const __half *src, float (&f)[NV])
{
    if constexpr (NV == 4) {
        const uint2 u = *reinterpret_cast<const uint2 *>(src);
        const float2 a = __half22float2(bits_h2(u.x)), c = __half22float2(bits_h2(u.y));
        f[0] = a.x; f[1] = a.y; f[2] = c.x; f[3] = c.y;
    } else if constexpr (NV == 2) {
        const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(src));
        f[0] = a.x; f[1] = a.y;
    } else {
        f[0] = __half2float(src[0]);
    }
}

// The fp16 residual window of one (sequence, kv head), taken by one more CTA
// of the chunk kernel's grid (it overlaps the chunks instead of following
// them): warp w takes tokens w, w + 8, ..., two at a time with both rows'
// loads issued first; lanes own 4 channels for the dot product (warp sum) and
// 4 coordinates for the values.  Writes part nsplit.  qf holds GQ * D floats,
// scratch the warps' merge.
template <int GQ>
__device__ __forceinline__ void ka_window(const KiviAttendParams &p, int bh, float *qf, unsigned char *scratch)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = bh / p.Hkv, h = bh - b * p.Hkv;
    int rl = p.res_lens ? __ldg(p.res_lens + b) : p.R;
    rl = rl < 0 ? 0 : (rl > p.R ? p.R : rl);
    const int nparts = p.nsplit + 1;
    if (rl == 0) return;  // the combine skips an empty window
    (void)ka_load_query<GQ, D>(p, b, h, qf, false);
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
    auto token = [&](uint2 ku, uint2 vu) {
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
    };
    for (int r = warp; r < rl; r += 2 * KA_WARPS) {
        const int r2 = r + KA_WARPS;
        const uint2 ku = __ldg(reinterpret_cast<const uint2 *>(kr + (size_t)r * D) + lane);
        const uint2 vu = __ldg(reinterpret_cast<const uint2 *>(vr + (size_t)r * D) + lane);
        uint2 ku2 = make_uint2(0u, 0u), vu2 = make_uint2(0u, 0u);
        if (r2 < rl) {
            ku2 = __ldg(reinterpret_cast<const uint2 *>(kr + (size_t)r2 * D) + lane);
            vu2 = __ldg(reinterpret_cast<const uint2 *>(vr + (size_t)r2 * D) + lane);
        }
        token(ku, vu);
        if (r2 < rl) token(ku2, vu2);
    }
    // l is already the warp's total (every lane holds the same sums)
    float *ms = reinterpret_cast<float *>(scratch);
    float *ls = ms + KA_WARPS * GQ;
    float *os = ls + KA_WARPS * GQ;
#pragma unroll
    for (int g = 0; g < GQ; ++g) {
        if (lane == 0) {
            ms[warp * GQ + g] = m[g];
            ls[warp * GQ + g] = l[g];
        }
        *reinterpret_cast<float4 *>(os + (warp * GQ + g) * D + 4 * lane) = make_float4(o[g][0], o[g][1], o[g][2], o[g][3]);
    }
    ka_merge_finish<GQ>(p, scratch, b, h, p.nsplit, nparts);
}

// The NV fp16 scales (or zeros) of one token, packed: halves 0, 1 in .x and
// 2, 3 in .y.
template <int NV>
__device__ __forceinline__ uint2 load_groups_raw(const __half *src)
{
    if constexpr (NV == 4) return *reinterpret_cast<const uint2 *>(src);
    else if constexpr (NV == 2) return make_uint2(*reinterpret_cast<const uint32_t *>(src), 0u);
    else return make_uint2((uint32_t)__half_as_ushort(src[0]), 0u);
}
// Group gr's scales of two tokens, as floats.
__device__ __forceinline__ float2 group_pair(uint2 a, uint2 b, int gr)
{
    const uint32_t wa = gr < 2 ? a.x : a.y, wb = gr < 2 ? b.x : b.y;
    const uint32_t sel = (gr & 1) ? 0x7632u : 0x5410u;  // the high or the low halves of both
    return __half22float2(bits_h2(__byte_perm(wa, wb, sel)));
}

// One chunk of the quantized tokens of one (sequence, kv head).
template <int BITS, int G, int GQ>
__global__ void __launch_bounds__(KA_WARPS * 32, GQ <= 4 ? 2 : 1)
    kivi_attend_kernel(const __grid_constant__ KiviAttendParams p)
{
    constexpr int STG = ka_stage(BITS, G);
    constexpr int KA_STAGES = ka_nst(BITS, G);
    constexpr int KW = BITS * 512;            // key words of a tile (bytes)
    constexpr int VW = KT * 16 * BITS;        // value words of a tile (bytes)
    constexpr int VS = KT * (D / G) * 2;      // value scales (or zeros) of a tile (bytes)
    constexpr int W = D * BITS / 32;          // value words per token
    constexpr int NV = D / G;                 // value groups per token
    constexpr int NT = (2 * GQ + 7) / 8;      // n-tiles of 8 (head, hi / lo) columns
    constexpr int MPQ = 8 / BITS;             // value m-tiles per 4 words of a token
    constexpr bool VPAIR = BITS < 4;          // value rows paired inside one byte (else split)
    constexpr uint32_t MASK = (1u << BITS) - 1u;
    extern __shared__ __align__(128) unsigned char smem[];
    float *qf = reinterpret_cast<float *>(smem);
    float *wb = qf + GQ * QS;
    unsigned char *stages = reinterpret_cast<unsigned char *>(wb + KA_WARPS * KT * GQ);
    uint64_t *bars = reinterpret_cast<uint64_t *>(stages + ka_region(BITS, G, GQ));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.y, split = blockIdx.x;
    if (split == p.nsplit) {  // the residual window's CTA (grid.x = nsplit + 1 when R > 0)
        ka_window<GQ>(p, bh, qf, stages);
        return;
    }
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
    const float pe = ka_load_query<GQ, QS>(p, b, h, qf, true);
    __syncthreads();

    // Fragment roles (m16n8k16), lane = 4 g8 + t4.  The lane's k entries
    // 2 t4, 2 t4 + 1, 2 t4 + 8, 2 t4 + 9 are channels 16 kt + 4 t4 + 0..3
    // (keys) or tokens 16 kt + t4 + 0, 4, 8, 12 (values).  Its B column g8 is
    // head 4 nt + g8 / 2, hi part for even g8, lo part for odd; its
    // accumulator columns 2 t4, 2 t4 + 1 are head 4 nt + t4, hi and lo.
    // Its operand rows g8 and g8 + 8 are entries 2 g8 and 2 g8 + 1 of the
    // m-tile's 16 (paired: both codes in one byte, one byte permute serves
    // both registers), or entries g8 and g8 + 8 (split: b = 4 values, whose
    // 16 coordinates span two words).  Codes enter as code * 2^shift; the
    // epilogue multiplies each row by 2^-shift.
    const int g8 = lane >> 2, t4 = lane & 3;
    const bool lo = (g8 & 1) != 0;
    const uint32_t mh = lo ? 0xFFFFFFFFu : 0xFFFFE000u, ml = lo ? 0xFFFFE000u : 0u;
    const int psh0 = (2 * g8 * BITS) & 7, psh1 = psh0 + BITS;
    const uint32_t pm0 = (MASK << psh0) * 0x10001u, pm1 = (MASK << psh1) * 0x10001u;
    uint32_t psel[2];  // by the parity of mt (only b = 1 depends on it)
#pragma unroll
    for (int par = 0; par < 2; ++par)
        psel[par] = (uint32_t)(((((16 * par + 2 * g8) * BITS) & 31) >> 3) * 0x1111 + 0x4400);
    const int kro = (2 * g8 * BITS) >> 5;  // key word row of entry 2 g8 past the m-tile's first
    const int ssh = (g8 * BITS) & 7;
    const uint32_t sm = (MASK << ssh) * 0x10001u;
    const uint32_t ssel = (uint32_t)((((g8 * BITS) & 31) >> 3) * 0x1111 + 0x4400);
    const float uk0 = __uint_as_float((uint32_t)(127 - psh0) << 23) * pe;
    const float uk1 = __uint_as_float((uint32_t)(127 - psh1) << 23) * pe;
    const float uv0 = __uint_as_float((uint32_t)(127 - (VPAIR ? psh0 : ssh)) << 23);
    const float uv1 = __uint_as_float((uint32_t)(127 - (VPAIR ? psh1 : ssh)) << 23);
    float *my_w = wb + warp * KT * GQ;  // weights [head][slot]

    float m[NT], l[NT], zb[NT][NV], acc_v[NT][8][4];
    float fsig = 30.0f;  // running exponent offset of the weights (non-increasing)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        m[nt] = NEG_INF;
        l[nt] = 0.0f;
#pragma unroll
        for (int gr = 0; gr < NV; ++gr) zb[nt][gr] = 0.0f;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc_v[nt][mt][j] = 0.0f;
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
        const uint32_t *kwords = reinterpret_cast<const uint32_t *>(sb);
        const __half *ksc = reinterpret_cast<const __half *>(sb + KW);
        const __half *kze = reinterpret_cast<const __half *>(sb + KW + 256);
        const uint32_t *vwords = reinterpret_cast<const uint32_t *>(sb + KW + 512);
        const __half *vsc = reinterpret_cast<const __half *>(sb + KW + 512 + VW);
        const __half *vze = reinterpret_cast<const __half *>(sb + KW + 512 + VW + VS);
        const bool full = n == KT;

        // ---- scores: S[token][(head, part)] = sum_c code[token][c] (q s)[c][(head, part)]
        float acc_k[NT][2][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc_k[nt][mt][j] = 0.0f;
#pragma unroll
        for (int kt = 0; kt < 8; ++kt) {
            const int c0 = 16 * kt + 4 * t4;
            const uint2 sv = *reinterpret_cast<const uint2 *>(ksc + c0);
            const float2 s01 = __half22float2(bits_h2(sv.x)), s23 = __half22float2(bits_h2(sv.y));
            uint32_t bk[NT][2];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int hb = 4 * nt + (g8 >> 1);
                float4 qv = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                if (GQ % 4 == 0 || hb < GQ) qv = *reinterpret_cast<const float4 *>(qf + hb * QS + c0);
                bk[nt][0] = split_pack(__fmul2_rn(make_float2(qv.x, qv.y), s01), mh, ml);
                bk[nt][1] = split_pack(__fmul2_rn(make_float2(qv.z, qv.w), s23), mh, ml);
            }
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
                const uint4 w4 = *reinterpret_cast<const uint4 *>(kwords + (mt * BITS / 2 + kro) * D + c0);
                const uint32_t x01 = __byte_perm(w4.x, w4.y, psel[mt]);
                const uint32_t x23 = __byte_perm(w4.z, w4.w, psel[mt]);
                const uint32_t a0 = code_h2(x01, pm0), a1 = code_h2(x01, pm1);
                const uint32_t a2 = code_h2(x23, pm0), a3 = code_h2(x23, pm1);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) mma_16816(acc_k[nt][mt], a0, a1, a2, a3, bk[nt][0], bk[nt][1]);
            }
        }
        // zero term sum_c q_c z_c of head 4 nt + (lane >> 3), channels
        // 4 (lane & 7) + 32 x, reduced over the 8 lanes of the head
        float bias[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int hz = 4 * nt + (lane >> 3), cz = 4 * (lane & 7);
            float bz = 0.0f;
            if (GQ % 4 == 0 || hz < GQ) {
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    const float4 q4 = *reinterpret_cast<const float4 *>(qf + hz * QS + cz + 32 * x);
                    const uint2 zu = *reinterpret_cast<const uint2 *>(kze + cz + 32 * x);
                    const float2 z01 = __half22float2(bits_h2(zu.x)), z23 = __half22float2(bits_h2(zu.y));
                    bz = fmaf(q4.x, z01.x, bz);
                    bz = fmaf(q4.y, z01.y, bz);
                    bz = fmaf(q4.z, z23.x, bz);
                    bz = fmaf(q4.w, z23.y, bz);
                }
            }
            bz += __shfl_xor_sync(FULL_MASK, bz, 1);
            bz += __shfl_xor_sync(FULL_MASK, bz, 2);
            bz += __shfl_xor_sync(FULL_MASK, bz, 4);
            bias[nt] = __shfl_sync(FULL_MASK, bz, 8 * t4) * pe;  // head 4 nt + t4
        }
        // exponent offset of the weights: with every value scale of the tile
        // below 2^(E + 1), weights up to 2^(14 - E) keep w s below 2^15 and
        // out of the fp16 subnormals (the offset enters the running max, so
        // it cancels in the normalisation).  The warp keeps the smallest
        // offset seen so far: a larger one would be as safe for this tile
        // but would move the running max (and rescale the sums) more often.
        {
            uint32_t mb = 0;
            if (4 * lane < KT * NV) {
                const uint2 su = *reinterpret_cast<const uint2 *>(vsc + 4 * lane);
                uint32_t hw[2] = {su.x & 0x7fff7fffu, su.y & 0x7fff7fffu};
                if (!full) {
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if ((4 * lane + j) / NV >= n) hw[j >> 1] &= (j & 1) ? 0x0000ffffu : 0xffff0000u;
                }
                const uint32_t mm = __vmaxu2(hw[0], hw[1]);
                mb = max(mm & 0xffffu, mm >> 16);
            }
            mb = __reduce_max_sync(FULL_MASK, mb);
            fsig = fminf(fsig, (float)min(14 - ((int)(mb >> 10) - 15), 30));
        }

        // ---- online softmax: this lane holds tokens 16 mt + 2 g8 + rh of head 4 nt + t4
        float w[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            float sc[4];
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int rh = 0; rh < 2; ++rh) {
                    const float a = acc_k[nt][mt][2 * rh] + acc_k[nt][mt][2 * rh + 1];
                    const float s = fmaf(a, rh ? uk1 : uk0, bias[nt]);
                    sc[2 * mt + rh] = (16 * mt + 2 * g8 + rh < n) ? s : NEG_INF;
                }
            float mx = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
            mx = fmaxf(mx, __shfl_xor_sync(FULL_MASK, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(FULL_MASK, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(FULL_MASK, mx, 16));
            const float cand = mx - fsig;
            if (cand > m[nt]) {
                const float f = exp2f(m[nt] - cand);
                l[nt] *= f;
#pragma unroll
                for (int gr = 0; gr < NV; ++gr) zb[nt][gr] *= f;
#pragma unroll
                for (int mt = 0; mt < 8; ++mt)
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc_v[nt][mt][j] *= f;
                m[nt] = cand;
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                w[nt][i] = exp2f(sc[i] - m[nt]);
                l[nt] += w[nt][i];
            }
            const int hh = 4 * nt + t4;
            if (GQ % 4 == 0 || hh < GQ) {
                // token 16 mt + r goes to slot 16 mt + 4 (r mod 4) + r / 4
#pragma unroll
                for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                    for (int rh = 0; rh < 2; ++rh) {
                        const int r = 2 * g8 + rh;
                        my_w[hh * KT + 16 * mt + 4 * (r & 3) + (r >> 2)] = w[nt][2 * mt + rh];
                    }
            }
        }
        // the value zeros' share sum_t w_t z_t, per head and value group
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int rh = 0; rh < 2; ++rh) {
                const int tok = 16 * mt + 2 * g8 + rh;
                float z[NV];
                load_groups<NV>(vze + tok * NV, z);
                if (!full && tok >= n) {
#pragma unroll
                    for (int gr = 0; gr < NV; ++gr) z[gr] = 0.0f;
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int gr = 0; gr < NV; ++gr) zb[nt][gr] = fmaf(w[nt][2 * mt + rh], z[gr], zb[nt][gr]);
            }
        __syncwarp();

        // ---- values: O[coord][(head, part)] += sum_t code[t][coord] (w s)[t][(head, part)]
#pragma unroll
        for (int kt = 0; kt < 2; ++kt) {
            uint2 sr[4];  // the NV fp16 scales of tokens 16 kt + t4 + 4 i
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int tok = 16 * kt + t4 + 4 * i;
                sr[i] = load_groups_raw<NV>(vsc + tok * NV);
                if (!full && tok >= n) sr[i] = make_uint2(0u, 0u);
            }
            float4 wv[NT];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int hb = 4 * nt + (g8 >> 1);
                wv[nt] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                if (GQ % 4 == 0 || hb < GQ) wv[nt] = *reinterpret_cast<const float4 *>(my_w + hb * KT + 16 * kt + 4 * t4);
            }
            uint32_t bv[NT][2];
#pragma unroll
            for (int qd = 0; qd < W / 4; ++qd) {
                uint4 vq[4];
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    vq[i] = *reinterpret_cast<const uint4 *>(vwords + (16 * kt + t4 + 4 * i) * W + 4 * qd);
#pragma unroll
                for (int mm = 0; mm < MPQ; ++mm) {
                    const int mt = qd * MPQ + mm;
                    if ((16 * mt) % G == 0) {  // first m-tile of value group gr: its (w s) columns
                        const int gr = 16 * mt / G;
                        const float2 s01 = group_pair(sr[0], sr[1], gr), s23 = group_pair(sr[2], sr[3], gr);
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            bv[nt][0] = split_pack(__fmul2_rn(make_float2(wv[nt].x, wv[nt].y), s01), mh, ml);
                            bv[nt][1] = split_pack(__fmul2_rn(make_float2(wv[nt].z, wv[nt].w), s23), mh, ml);
                        }
                    }
                    uint32_t a0, a1, a2, a3;
                    if constexpr (VPAIR) {
                        const int o = mt * BITS / 2 - 4 * qd;  // word of coordinates 16 mt + 2 g8, + 1
                        const uint32_t x01 = __byte_perm(quad_at(vq[0], o), quad_at(vq[1], o), psel[mt & 1]);
                        const uint32_t x23 = __byte_perm(quad_at(vq[2], o), quad_at(vq[3], o), psel[mt & 1]);
                        a0 = code_h2(x01, pm0); a1 = code_h2(x01, pm1); a2 = code_h2(x23, pm0); a3 = code_h2(x23, pm1);
                    } else {
                        const int o0 = 2 * mt - 4 * qd, o1 = o0 + 1;  // words of coordinates 16 mt + g8, + 8
                        a0 = code_h2(__byte_perm(quad_at(vq[0], o0), quad_at(vq[1], o0), ssel), sm);
                        a1 = code_h2(__byte_perm(quad_at(vq[0], o1), quad_at(vq[1], o1), ssel), sm);
                        a2 = code_h2(__byte_perm(quad_at(vq[2], o0), quad_at(vq[3], o0), ssel), sm);
                        a3 = code_h2(__byte_perm(quad_at(vq[2], o1), quad_at(vq[3], o1), ssel), sm);
                    }
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) mma_16816(acc_v[nt][mt], a0, a1, a2, a3, bv[nt][0], bv[nt][1]);
                }
            }
        }

        __syncwarp();
        fence_proxy_async_smem();
        if (t + KA_STAGES * KA_WARPS < ntiles) issue(t + KA_STAGES * KA_WARPS, st);
    }

    // totals over the 8 row lanes of each head, then the head's outputs:
    // (hi + lo) 2^-shift + the zeros' share
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int off = 4; off <= 16; off <<= 1) {
            l[nt] += __shfl_xor_sync(FULL_MASK, l[nt], off);
#pragma unroll
            for (int gr = 0; gr < NV; ++gr) zb[nt][gr] += __shfl_xor_sync(FULL_MASK, zb[nt][gr], off);
        }
    __syncthreads();  // every warp is done with its stages: they hold the merge now
    float *ms = reinterpret_cast<float *>(stages);
    float *ls = ms + KA_WARPS * GQ;
    float *os = ls + KA_WARPS * GQ;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int hh = 4 * nt + t4;
        if (GQ % 4 == 0 || hh < GQ) {
            if (g8 == 0) {
                ms[warp * GQ + hh] = m[nt];
                ls[warp * GQ + hh] = l[nt];
            }
            float *o = os + (warp * GQ + hh) * D;
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                const float z = zb[nt][16 * mt / G];
                const int d0 = VPAIR ? 16 * mt + 2 * g8 : 16 * mt + g8;
                const int d1 = VPAIR ? d0 + 1 : d0 + 8;
                o[d0] = fmaf(acc_v[nt][mt][0] + acc_v[nt][mt][1], uv0, z);
                o[d1] = fmaf(acc_v[nt][mt][2] + acc_v[nt][mt][3], uv1, z);
            }
        }
    }
    ka_merge_finish<GQ>(p, stages, b, h, split, nparts);
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
    dim3 grid(nparts, p.B * p.Hkv);  // the window's part is one more CTA per (sequence, kv head)
    kern<<<grid, KA_WARPS * 32, smem, stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
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
