// attend.cu - decode-time attention over a TurboQuantRVQ key cache (sm_103a).
//
// Method (VeloxQuant-MLX blog, tag "turboquant", "Kernel 5: Fused RVQ Decode
// + Attend — Online Softmax Without Materializing K"): keys are decoded from
// their two code streams on the fly, the softmax is taken online and values
// are accumulated, so the decoded keys never reach memory.  Because H/sqrt(D)
// is symmetric and orthogonal,
//   q . k_s = n_s (H q / sqrt(D)) . (c1[i1] + c2[i2]),
// so the query is rotated once and every key is scored in the rotated domain
// straight from its codes, with no inverse transform per key.
//
// Design.  The valid tokens of each (sequence, kv head) are cut into chunks of
// a fixed number of keys; one CTA of 8 warps takes one chunk, so the grid is
// balanced whatever the mix of cache lengths.  The GQ = Hq / Hkv query heads
// of a kv head are served together, so each key and value row is read once.
// Each warp streams its own 16-key tiles: TMA lands the tile's value rows
// (two 64-coordinate boxes, 128-byte swizzled) and the bulk-copy engine both
// code streams in one of two shared-memory stages per warp while the warp
// works on the other.  Both sums of a tile are dense products on the tensor
// cores (16 x 8 x 16 mma.sync, fp16 operands, fp32 accumulation):
//   scores   S[key][(head, hi/lo)] = sum_c y[key][c] Q[c][(head, hi/lo)]: y is
//            the decoded rotated key, one shuffle of a (hi, lo) fp16 pair per
//            coordinate from the merged c1 + c2 table (two tables at b = 4),
//            Q the rotated query carried as two fp16 columns per head (built
//            once per CTA); both scaled by powers of two into fp16 range;
//   softmax  one head per lane (its two keys), tile maximum by three shuffles;
//   values   O[coord][(head, hi/lo)] += sum_k V[k][coord] w[k][(head, hi/lo)],
//            the fp16 values read transposed from the swizzled boxes
//            (ldmatrix), each weight carried as two fp16 columns.
// Every float factor keeps about 21 bits through its hi/lo split.
// Warps, then CTAs (the chunks, through the caller's workspace and a combine
// kernel), are merged at the end.  Softmax arithmetic is in base 2 (the query
// carries scale * log2(e)).
#include <cuda_fp16.h>


#include "device_common.cuh"
#include "launch.h"

namespace vq {

namespace {

VQ_DEFINE_ERROR_WORD(g_at_err);

// Scratch for the split partials of vq_rvq_attend_noalloc (no caller
// workspace); one array per device, in the module's static device memory.
static __device__ __align__(256) float g_at_scratch[VQ_ATTEND_SCRATCH_BYTES / sizeof(float)];

constexpr int D = 128;
constexpr int AT_WARPS = 8;
constexpr int TK = 32;    // chunk sizes are multiples of 32 keys
constexpr int TILE = 16;  // keys per warp tile: one 16-row m-tile of the score product
constexpr int AT_STAGES = 2;
constexpr float NEG_INF = -__builtin_huge_valf();

template <int BITS>
struct AtTile {
    static constexpr int W = D * BITS / 32;       // code words per key and stream
    static constexpr int VAL = TILE * D * 2;      // value rows of a tile: two 64-coordinate boxes
    static constexpr int COD = TILE * W * 4;      // one code stream of a tile
    static constexpr int STAGE = (VAL + 2 * COD + 1023) / 1024 * 1024;  // boxes stay 1024-aligned
};

constexpr int WS = TILE + 8;  // weights row stride (floats) per head: 4 heads on distinct banks
constexpr float SIG = 14.0f;  // exponent offset of the weights (w <= 2^14, never fp16-subnormal)
constexpr int QPAD = 4;       // the query's coordinates 64..127 sit 16 bytes further (other banks)

template <int BITS, int GQ>
constexpr int at_smem()
{
    return 1024                                         // alignment slack (128-byte swizzle)
           + AT_WARPS * AT_STAGES * AtTile<BITS>::STAGE // stages (multiples of 1024 bytes)
           + (D * GQ + QPAD) * 4                        // rotated query [c][g]
           + ((2 * GQ + 7) / 8) * 8 * 32 * 8            // its B fragments [nt][kt][lane] (uint2)
           + AT_WARPS * GQ * WS * 4                     // weights [warp][g][key]
           + AT_WARPS * AT_STAGES * 8;                  // mbarriers
}

__device__ __forceinline__ float2 f2(float a, float b) { return make_float2(a, b); }
__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }

// The fp16 pair of this lane's part of (w0, w1): hi lanes (mh = ~0x1fff,
// ml = 0) take w with its mantissa cut to fp16's 10 bits (exact in fp16), lo
// lanes (mh = ~0, ml = ~0x1fff) the rest, rounded to fp16; the two columns of
// one head together carry w to about 21 bits.
__device__ __forceinline__ uint32_t split_pack(float2 u, uint32_t mh, uint32_t ml)
{
    const uint32_t ux = __float_as_uint(u.x), uy = __float_as_uint(u.y);
    const float2 a = f2(__uint_as_float(ux & mh), __uint_as_float(uy & mh));
    const float2 c = f2(__uint_as_float((ux & ml) ^ 0x80000000u), __uint_as_float((uy & ml) ^ 0x80000000u));
    return h2_bits(__float22half2_rn(__fadd2_rn(a, c)));
}

// (fp16(x), fp16(x - fp16(x))) in the low and high halves: x to about 22 bits.
__device__ __forceinline__ __half2 hilo(float x)
{
    const __half hi = __float2half_rn(x);
    return __halves2half2(hi, __float2half_rn(x - __half2float(hi)));
}

// Four 8 x 8 fp16 matrices from shared memory, transposed (lane i supplies the
// row address of matrix i / 8).
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
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

template <int BITS, int GQ>
__global__ void __launch_bounds__(AT_WARPS * 32, 2) rvq_attend_kernel(const __grid_constant__ RvqAttendParams p)
{
    using T = AtTile<BITS>;
    constexpr int W = T::W;
    constexpr int L = 1 << BITS;
    constexpr int NT = (2 * GQ + 7) / 8;  // value n-tiles of 8 (head, hi / lo) columns
    extern __shared__ __align__(128) unsigned char smem_raw[];
    unsigned char *stages = smem_1k(smem_raw);
    float *qs = reinterpret_cast<float *>(stages + AT_WARPS * AT_STAGES * T::STAGE);
    uint2 *bqs = reinterpret_cast<uint2 *>(qs + D * GQ + QPAD);  // [nt][kt][lane]
    float *wb = reinterpret_cast<float *>(bqs + NT * 8 * 32);
    uint64_t *bars = reinterpret_cast<uint64_t *>(wb + AT_WARPS * GQ * WS);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.y, split = blockIdx.x;
    const int b = bh / p.Hkv, h = bh - b * p.Hkv;
    int len = p.lens ? __ldg(p.lens + b) : p.S_cap;
    len = len < 0 ? 0 : (len > p.S_cap ? p.S_cap : len);
    const int s0 = split * p.chunk;
    if (s0 >= len && !(split == 0 && p.nsplit == 1)) return;  // no keys: the combine skips this chunk
    const int s1 = min(len, s0 + p.chunk);
    const int ntiles = s1 > s0 ? (s1 - s0 + TILE - 1) / TILE : 0;

    unsigned char *my_st = stages + warp * AT_STAGES * T::STAGE;
    uint64_t *my_bar = bars + warp * AT_STAGES;
    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < AT_STAGES; ++s) mbar_init(&my_bar[s], 1);
        fence_mbar_init();
    }
    __syncwarp();
    const size_t kbase = (size_t)bh * p.S_cap;
    const uint64_t pol = l2_policy_evict_first();
    auto issue = [&](int t, int st) {
        if (lane == 0) {
            const int k0 = s0 + t * TILE;
            const int n = min(TILE, s1 - k0);
            unsigned char *dst = my_st + st * T::STAGE;
            // value rows: two boxes of 64 coordinates x 16 rows, 128-byte swizzle
            // (rows past the tensor are zero-filled, every box counts in full)
            mbar_arrive_expect_tx(&my_bar[st], (uint32_t)(T::VAL + n * 2 * W * 4));
            tma_load_2d(dst, &p.tmv, 0, (int)(kbase + k0), &my_bar[st], pol);
            tma_load_2d(dst + T::VAL / 2, &p.tmv, 64, (int)(kbase + k0), &my_bar[st], pol);
            bulk_g2s(dst + T::VAL, p.p1 + (kbase + k0) * W, (uint32_t)(n * W * 4), &my_bar[st], pol);
            bulk_g2s(dst + T::VAL + T::COD, p.p2 + (kbase + k0) * W, (uint32_t)(n * W * 4), &my_bar[st], pol);
        }
    };
#pragma unroll
    for (int s = 0; s < AT_STAGES; ++s) {
        const int t = warp + s * AT_WARPS;
        if (t < ntiles) issue(t, s);
    }

    // rotated, pre-scaled query of the GQ heads: warp g transforms head g
    if (warp < GQ) {
        const __half *qh = static_cast<const __half *>(p.q) + ((size_t)b * p.Hq + (size_t)h * GQ + warp) * D;
        uint2 raw = *reinterpret_cast<const uint2 *>(qh + 4 * lane);
        if (p.has_sgn) {
            // randomised signs: the query is rotated by H diag(s) like the keys
            raw.x ^= half2_sign_mask(sign_pair(p.sgn, 4 * lane));
            raw.y ^= half2_sign_mask(sign_pair(p.sgn, 4 * lane + 2));
        }
        const __half2 h01 = *reinterpret_cast<const __half2 *>(&raw.x);
        const __half2 h23 = *reinterpret_cast<const __half2 *>(&raw.y);
        float a[4] = {__low2float(h01), __high2float(h01), __low2float(h23), __high2float(h23)};
        float t0 = a[0] + a[1], t1 = a[0] - a[1], t2 = a[2] + a[3], t3 = a[2] - a[3];
        a[0] = t0 + t2; a[1] = t1 + t3; a[2] = t0 - t2; a[3] = t1 - t3;
#pragma unroll
        for (int m = 1; m < 32; m <<= 1) {
            const bool upper = (lane & m) != 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float o = __shfl_xor_sync(FULL_MASK, a[j], m);
                a[j] = upper ? (o - a[j]) : (a[j] + o);
            }
        }
        float amax = 0.0f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            a[j] *= p.qscale;
            qs[(4 * lane + j) * GQ + (lane >= 16 ? QPAD : 0) + warp] = a[j];
            amax = fmaxf(amax, fabsf(a[j]));
        }
        amax = __uint_as_float(__reduce_max_sync(FULL_MASK, __float_as_uint(amax)));
        if (lane == 0) wb[warp] = amax;  // the weights area is free until the tile loop
    }
    __syncthreads();

    // Scores on the tensor cores: S[key][(head, hi/lo)] = sum_c y[key][c]
    // Q[c][(head, hi/lo)], y the decoded rotated key (table value, fp16 hi +
    // lo), Q the rotated query scaled by 2^eq (fp16 hi + lo columns).  Both
    // scales are powers of two that bring the largest |entry| below 2^15.
    int eq = 0, et = 0;
    {
        float qm = 0.0f;
        for (int g = 0; g < GQ; ++g) qm = fmaxf(qm, wb[g]);
        if (qm > 0.0f && qm < 1.0e30f) eq = 14 - ((int)((__float_as_uint(qm) >> 23) & 0xffu) - 127);
        eq = max(-100, min(eq, 100));
    }
    // lane holds table entry lane mod 2^(2b) (merged c1 + c2, b <= 2) or the
    // two stage tables' entries lane mod 16 (b = 4), scaled by 2^et
    const float ty1 = BITS == 4 ? p.c1[lane & (L - 1)] : p.c1[lane & (L - 1)] + p.c2[(lane >> BITS) & (L - 1)];
    const float ty2 = BITS == 4 ? p.c2[lane & (L - 1)] : 0.0f;
    {
        const float tm = __uint_as_float(__reduce_max_sync(FULL_MASK, __float_as_uint(fmaxf(fabsf(ty1), fabsf(ty2)))));
        if (tm > 0.0f && tm < 1.0e30f) et = 14 - ((int)((__float_as_uint(tm) >> 23) & 0xffu) - 127);
        et = max(-100, min(et, 100));
    }
    const float tsc = ldexpf(1.0f, et);
    const uint32_t th1 = h2_bits(hilo(ty1 * tsc)), th2 = h2_bits(hilo(ty2 * tsc));
    const float sunscale = ldexpf(1.0f, -(et + eq));  // exact: undoes both scales

    // B fragments of the query (built once per CTA, read per k-tile): lane
    // (g8, t4) of n-tile nt holds column g8 = (head 4 nt + g8 / 2, hi / lo)
    // at coordinates 16 kt + 4 t4 + {0, 1} and + {2, 3}
    {
        const int g8 = lane >> 2, t4 = lane & 3;
        const bool lo = (g8 & 1) != 0;
        const uint32_t mh = lo ? 0xFFFFFFFFu : 0xFFFFE000u, ml = lo ? 0xFFFFE000u : 0u;
        const float qsc = ldexpf(1.0f, eq);
        for (int i = warp; i < NT * 8; i += AT_WARPS) {
            const int nt = i >> 3, kt = i & 7;
            const int hb = 4 * nt + (g8 >> 1);
            float u[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            if (hb < GQ) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int c = 16 * kt + 4 * t4 + j;
                    u[j] = qs[c * GQ + (c >= 64 ? QPAD : 0) + hb] * qsc;
                }
            }
            bqs[i * 32 + lane] = make_uint2(split_pack(f2(u[0], u[1]), mh, ml), split_pack(f2(u[2], u[3]), mh, ml));
        }
    }
    __syncthreads();  // the query maxima in wb are read; the weights may overwrite them

    float *my_w = wb + warp * GQ * WS;  // weights [g][key]

    // Values on the tensor cores: O[coord][(head, part)] += sum_k V[k][coord]
    // w[k][(head, part)], 16 x 8 x 16 tiles.  Lane = 4 g8 + t4: its
    // accumulator rows are coordinates 16 mt + g8 and + 8, its columns
    // 2 t4, 2 t4 + 1 head 4 nt + t4, hi and lo; its B column g8 is head
    // 4 nt + g8 / 2, hi part for even g8, lo part for odd.
    const int g8 = lane >> 2, t4 = lane & 3;
    const bool lo = (g8 & 1) != 0;
    const uint32_t mh = lo ? 0xFFFFFFFFu : 0xFFFFE000u, ml = lo ? 0xFFFFE000u : 0u;
    float m[NT], l[NT];  // running max (with the SIG offset) and sum of head 4 nt + t4
    float acc[NT][8][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        m[nt] = NEG_INF;
        l[nt] = 0.0f;
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[nt][mt][j] = 0.0f;

    for (int it = 0;; ++it) {
        const int t = warp + it * AT_WARPS;
        if (t >= ntiles) break;
        const int st = it % AT_STAGES;
        const int k0 = s0 + t * TILE;
        const int n = min(TILE, s1 - k0);
        const bool va = g8 < n, vb = g8 + 8 < n;  // this lane's two keys (rows g8, g8 + 8)
        const float na = va ? __ldg(p.norms + kbase + k0 + g8) : 0.0f;
        const float nb = vb ? __ldg(p.norms + kbase + k0 + g8 + 8) : 0.0f;
        const bool ok = mbar_wait_bounded(&my_bar[st], (uint32_t)(it / AT_STAGES) & 1u);
        if (!__all_sync(FULL_MASK, ok)) {
            if (lane == 0) atomicOr(&g_at_err, (unsigned)VQ_DEVERR_WAIT_TIMEOUT);
            for (int k = 1; k < AT_STAGES; ++k) {
                const int it2 = it + k;
                if (warp + it2 * AT_WARPS < ntiles)
                    (void)mbar_wait_bounded(&my_bar[it2 % AT_STAGES], (uint32_t)(it2 / AT_STAGES) & 1u);
            }
            break;
        }
        const unsigned char *sb = my_st + st * T::STAGE;

        // scores: rows are the tile's keys g8, g8 + 8; the lane's k entries
        // 2 t4, 2 t4 + 1, 2 t4 + 8, 2 t4 + 9 are coordinates 16 kt + 4 t4 + 0..3
        float accs[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int j = 0; j < 4; ++j) accs[nt][j] = 0.0f;
        {
            const uint32_t *c1a = reinterpret_cast<const uint32_t *>(sb + T::VAL) + g8 * W;
            const uint32_t *c2a = reinterpret_cast<const uint32_t *>(sb + T::VAL + T::COD) + g8 * W;
            const uint32_t *c1b = c1a + 8 * W, *c2b = c2a + 8 * W;
#pragma unroll
            for (int kt = 0; kt < 8; ++kt) {
                uint32_t ah[4], al[4];  // A fragments (hi and lo parts of y)
                uint32_t ah2[4], al2[4];  // b = 4: the stage-2 table's parts
                auto rows = [&](const uint32_t *p1w, const uint32_t *p2w, int r) {
                    // r = 0: row g8 (registers 0, 2); r = 1: row g8 + 8 (registers 1, 3)
                    if constexpr (BITS == 4) {
                        const uint32_t x1 = p1w[2 * kt + (t4 >> 1)], x2 = p2w[2 * kt + (t4 >> 1)];
                        const int sh = 16 * (t4 & 1);
                        uint32_t v1[4], v2[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            v1[j] = __shfl_sync(FULL_MASK, th1, (int)(x1 >> (sh + 4 * j)));
                            v2[j] = __shfl_sync(FULL_MASK, th2, (int)(x2 >> (sh + 4 * j)));
                        }
                        ah[r] = __byte_perm(v1[0], v1[1], 0x5410); al[r] = __byte_perm(v1[0], v1[1], 0x7632);
                        ah[r + 2] = __byte_perm(v1[2], v1[3], 0x5410); al[r + 2] = __byte_perm(v1[2], v1[3], 0x7632);
                        ah2[r] = __byte_perm(v2[0], v2[1], 0x5410); al2[r] = __byte_perm(v2[0], v2[1], 0x7632);
                        ah2[r + 2] = __byte_perm(v2[2], v2[3], 0x5410); al2[r + 2] = __byte_perm(v2[2], v2[3], 0x7632);
                    } else {
                        // merged index i1 | i2 << BITS: even coordinates from me, odd from mo
                        constexpr uint32_t CM = BITS == 2 ? 0x33333333u : 0x55555555u;
                        constexpr int E = 32 / BITS;
                        const int wi = (16 * kt) / E;
                        const int base = (16 * kt) % E + 4 * t4;
                        const uint32_t x1 = p1w[wi], x2 = p2w[wi];
                        const uint32_t me = (x1 & CM) | ((x2 << BITS) & ~CM);
                        const uint32_t mo = ((x1 >> BITS) & CM) | (x2 & ~CM);
                        const uint32_t v0 = __shfl_sync(FULL_MASK, th1, (int)(me >> (base * BITS)));
                        const uint32_t v1 = __shfl_sync(FULL_MASK, th1, (int)(mo >> (base * BITS)));
                        const uint32_t v2 = __shfl_sync(FULL_MASK, th1, (int)(me >> ((base + 2) * BITS)));
                        const uint32_t v3 = __shfl_sync(FULL_MASK, th1, (int)(mo >> ((base + 2) * BITS)));
                        ah[r] = __byte_perm(v0, v1, 0x5410); al[r] = __byte_perm(v0, v1, 0x7632);
                        ah[r + 2] = __byte_perm(v2, v3, 0x5410); al[r + 2] = __byte_perm(v2, v3, 0x7632);
                    }
                };
                rows(c1a, c2a, 0);
                rows(c1b, c2b, 1);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const uint2 bq = bqs[(nt * 8 + kt) * 32 + lane];
                    mma_16816(accs[nt], ah[0], ah[1], ah[2], ah[3], bq.x, bq.y);
                    mma_16816(accs[nt], al[0], al[1], al[2], al[3], bq.x, bq.y);
                    if constexpr (BITS == 4) {
                        mma_16816(accs[nt], ah2[0], ah2[1], ah2[2], ah2[3], bq.x, bq.y);
                        mma_16816(accs[nt], al2[0], al2[1], al2[2], al2[3], bq.x, bq.y);
                    }
                }
            }
        }

        // online softmax: this lane holds keys g8, g8 + 8 of head 4 nt + t4;
        // the running maximum carries an offset of SIG so the weights reach
        // up to 2^SIG (it cancels in the merge)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const float sa = va ? (accs[nt][0] + accs[nt][1]) * sunscale * na : NEG_INF;
            const float sbb = vb ? (accs[nt][2] + accs[nt][3]) * sunscale * nb : NEG_INF;
            float mx = fmaxf(sa, sbb);
            mx = fmaxf(mx, __shfl_xor_sync(FULL_MASK, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(FULL_MASK, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(FULL_MASK, mx, 16));
            const float cand = mx - SIG;
            if (cand > m[nt]) {  // uniform over the 8 lanes of the head
                const float f = exp2f(m[nt] - cand);
                l[nt] *= f;
#pragma unroll
                for (int mt = 0; mt < 8; ++mt)
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[nt][mt][j] *= f;
                m[nt] = cand;
            }
            const float wa = exp2f(sa - m[nt]), wbb = exp2f(sbb - m[nt]);
            l[nt] += wa + wbb;
            const int hh = 4 * nt + t4;
            if (GQ % 4 == 0 || hh < GQ) {
                my_w[hh * WS + g8] = wa;
                my_w[hh * WS + g8 + 8] = wbb;
            }
        }
        __syncwarp();

        // values: the weight columns, then 8 blocks of 16 coordinates read
        // transposed from the swizzled value boxes
        const uint32_t vbase = smem_u32(sb);
#pragma unroll
        for (int kt = 0; kt < TILE / 16; ++kt) {
            uint32_t bv[NT][2];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int hb = 4 * nt + (g8 >> 1);
                float2 w01 = f2(0.0f, 0.0f), w89 = f2(0.0f, 0.0f);
                if (GQ % 4 == 0 || hb < GQ) {
                    w01 = *reinterpret_cast<const float2 *>(my_w + hb * WS + 16 * kt + 2 * t4);
                    w89 = *reinterpret_cast<const float2 *>(my_w + hb * WS + 16 * kt + 2 * t4 + 8);
                }
                bv[nt][0] = split_pack(w01, mh, ml);
                bv[nt][1] = split_pack(w89, mh, ml);
            }
            // keys past n hold stale rows: mask their halves out of the operands
            uint32_t ka = 0xFFFFFFFFu, kb = 0xFFFFFFFFu;
            if (n < TILE) {
                const int k = 16 * kt + 2 * t4;
                ka = (k < n ? 0x0000FFFFu : 0u) | (k + 1 < n ? 0xFFFF0000u : 0u);
                kb = (k + 8 < n ? 0x0000FFFFu : 0u) | (k + 9 < n ? 0xFFFF0000u : 0u);
            }
            // lane i of the ldmatrix supplies row (key) 16 kt + 8 (i / 16) + i % 8 of
            // 16-byte chunk 2 (mt % 4) + (i / 8) % 2 of box mt / 4
            const int key = 16 * kt + 8 * (lane >> 4) + (lane & 7);
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                const int c = 2 * (mt & 3) + ((lane >> 3) & 1);
                const uint32_t addr = vbase + (uint32_t)((mt >> 2) * (T::VAL / 2)) + swz128(key, c);
                uint32_t a0, a1, a2, a3;
                ldsm_x4_t(addr, a0, a1, a2, a3);
                a0 &= ka; a1 &= ka; a2 &= kb; a3 &= kb;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) mma_16816(acc[nt][mt], a0, a1, a2, a3, bv[nt][0], bv[nt][1]);
            }
        }

        // the stage and the weights are consumed: recycle the stage
        __syncwarp();
        fence_proxy_async_smem();
        if (t + AT_STAGES * AT_WARPS < ntiles) issue(t + AT_STAGES * AT_WARPS, st);
    }

    // per-warp sums, then merge the warps through shared memory (the stages
    // are free: every copy this CTA issued has been waited for)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int off = 4; off <= 16; off <<= 1) l[nt] += __shfl_xor_sync(FULL_MASK, l[nt], off);
    __syncthreads();
    float *ms = reinterpret_cast<float *>(stages);
    float *ls = ms + AT_WARPS * GQ;
    float *os = ls + AT_WARPS * GQ;  // [warp][g][D]
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
                o[16 * mt + g8] = acc[nt][mt][0] + acc[nt][mt][1];
                o[16 * mt + g8 + 8] = acc[nt][mt][2] + acc[nt][mt][3];
            }
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < GQ * D; i += blockDim.x) {
        const int g = i / D, d = i - g * D;
        float M = NEG_INF;
#pragma unroll
        for (int k = 0; k < AT_WARPS; ++k) M = fmaxf(M, ms[k * GQ + g]);
        float Ls = 0.0f, O = 0.0f;
#pragma unroll
        for (int k = 0; k < AT_WARPS; ++k) {
            const float mk = ms[k * GQ + g];
            const float f = (mk == NEG_INF) ? 0.0f : exp2f(mk - M);
            Ls = fmaf(ls[k * GQ + g], f, Ls);
            O = fmaf(os[(k * GQ + g) * D + d], f, O);
        }
        const int hq = h * GQ + g;
        if (p.nsplit == 1) {
            static_cast<__half *>(p.out)[((size_t)b * p.Hq + hq) * D + d] =
                __float2half_rn(Ls > 0.0f ? O / Ls : 0.0f);
        } else {
            float *wp = p.ws + (((size_t)b * p.Hq + hq) * p.nsplit + split) * AT_PART;
            if (d == 0) {
                wp[0] = M;
                wp[1] = Ls;
            }
            wp[2 + d] = O;
        }
    }
}

// Combine the chunks of one (sequence, query head): 128 threads, one per
// coordinate; only the chunks that hold keys were written.
__global__ void __launch_bounds__(D) rvq_attend_combine_kernel(const __grid_constant__ RvqAttendParams p)
{
    const int bq = blockIdx.x, d = threadIdx.x;
    const int b = bq / p.Hq;
    int len = p.lens ? __ldg(p.lens + b) : p.S_cap;
    len = len < 0 ? 0 : (len > p.S_cap ? p.S_cap : len);
    const int nv = (len + p.chunk - 1) / p.chunk;
    const float *wp = p.ws + (size_t)bq * p.nsplit * AT_PART;
    float M = NEG_INF;
    for (int s = 0; s < nv; ++s) M = fmaxf(M, wp[(size_t)s * AT_PART]);
    float Ls = 0.0f, O = 0.0f;
    for (int s = 0; s < nv; ++s) {
        const float ms = wp[(size_t)s * AT_PART];
        const float f = (ms == NEG_INF) ? 0.0f : exp2f(ms - M);
        Ls = fmaf(wp[(size_t)s * AT_PART + 1], f, Ls);
        O = fmaf(wp[(size_t)s * AT_PART + 2 + d], f, O);
    }
    static_cast<__half *>(p.out)[(size_t)bq * D + d] = __float2half_rn(Ls > 0.0f ? O / Ls : 0.0f);
}

template <int BITS, int GQ>
cudaError_t launch_at(const RvqAttendParams &p, cudaStream_t stream)
{
    RvqAttendParams q = p;
    const uint64_t rows = (uint64_t)p.B * p.Hkv * p.S_cap;
    if (rows > 0x7fffffffULL) return cudaErrorInvalidValue;  // TMA row coordinates are 32-bit
    if (rows > 0) {
        const uint64_t dims[2] = {(uint64_t)D, rows};
        const uint64_t strides[1] = {(uint64_t)D * 2};
        const uint32_t box[2] = {64u, (uint32_t)TILE};
        if (!encode_tmap_f16(&q.tmv, p.v, 2, dims, strides, box, true, true)) return cudaErrorInvalidValue;
    }
    auto kern = rvq_attend_kernel<BITS, GQ>;
    constexpr int smem = at_smem<BITS, GQ>();
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    dim3 grid(q.nsplit, q.B * q.Hkv);
    kern<<<grid, AT_WARPS * 32, smem, stream>>>(q);
    e = cudaGetLastError();
    if (e != cudaSuccess || q.nsplit == 1) return e;
    rvq_attend_combine_kernel<<<q.B * q.Hq, D, 0, stream>>>(q);
    return cudaGetLastError();
}

template <int BITS>
cudaError_t dispatch_at(const RvqAttendParams &p, cudaStream_t stream)
{
    switch (p.Hq / p.Hkv) {
    case 1: return launch_at<BITS, 1>(p, stream);
    case 2: return launch_at<BITS, 2>(p, stream);
    case 4: return launch_at<BITS, 4>(p, stream);
    case 8: return launch_at<BITS, 8>(p, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

void rvq_attend_plan(int B, int Hkv, int S_cap, int *nsplit, int *chunk)
{
    // chunks of 256 .. 2048 keys (a multiple of the 32-key tile), sized for
    // about eight waves of one CTA per SM over full caches
    const long long units = (long long)B * Hkv;
    if (units <= 0 || S_cap <= 0) {
        *nsplit = 1;
        *chunk = TK;
        return;
    }
    long long c = (units * S_cap + 8LL * sm_count() - 1) / (8LL * sm_count());
    c = (c + TK - 1) / TK * TK;
    c = c < 256 ? 256 : (c > 2048 ? 2048 : c);
    int n = (int)((S_cap + c - 1) / c);
    if (n <= 1) {
        *nsplit = 1;
        *chunk = (S_cap + TK - 1) / TK * TK;
        return;
    }
    *nsplit = n;
    *chunk = (int)c;
}

void rvq_attend_plan_fit(int S_cap, int max_splits, int *nsplit, int *chunk)
{
    // the largest number of chunks that fits: chunk = ceil(S_cap / max_splits)
    if (max_splits < 2 || S_cap <= TK) {
        *nsplit = 1;
        *chunk = (S_cap + TK - 1) / TK * TK;
        if (*chunk < TK) *chunk = TK;
        return;
    }
    int c = (S_cap + max_splits - 1) / max_splits;
    c = (c + TK - 1) / TK * TK;
    *chunk = c;
    *nsplit = (S_cap + c - 1) / c;
}

cudaError_t launch_rvq_attend(const RvqAttendParams &p, int bits, cudaStream_t stream)
{
    if (p.B <= 0 || p.Hq <= 0) return cudaSuccess;
    switch (bits) {
    case 1: return dispatch_at<1>(p, stream);
    case 2: return dispatch_at<2>(p, stream);
    case 4: return dispatch_at<4>(p, stream);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t attend_static_scratch(void **ptr, size_t *bytes)
{
    // The symbol's device address on the current device, looked up on every
    // call (a table lookup once the module is loaded): a cached address would
    // outlive a cudaDeviceReset, after which the array lives elsewhere.
    void *addr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&addr, g_at_scratch);
    if (e != cudaSuccess) return e;
    *ptr = addr;
    *bytes = sizeof(g_at_scratch);
    return cudaSuccess;
}

cudaError_t attend_take_device_error(unsigned *bits, cudaStream_t stream)
{
    *bits = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(bits, g_at_err, sizeof(unsigned), 0, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    if (*bits) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbolAsync(g_at_err, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice, stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    }
    return e;
}

}  // namespace vq
