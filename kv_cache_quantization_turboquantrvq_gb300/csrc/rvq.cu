// rvq.cu - TurboQuantRVQ encode+pack and unpack+dequant kernels for sm_103a.
//
// The encoders' device code (method, design and exactness notes) is in
// rvq_encode.cuh; here are their kernels (one persistent CTA per SM, each
// running the shared body over its share of the rows), the decoder and the
// launchers.
#include <cuda_fp16.h>

#include "device_common.cuh"
#include "launch.h"

namespace vq {
VQ_DEFINE_ERROR_WORD(g_rvq_err);
}  // namespace vq

#define VQ_RVQ_ERR g_rvq_err
#include "rvq_encode.cuh"
#include "tcgen05.cuh"

namespace vq {

namespace {

// SGN: the randomised-sign rotation (a separate instantiation, so that the
// plain rotation carries no per-row test).
template <int BITS, int MODE, bool SGN>
__global__ void __launch_bounds__(enc_warps(BITS, MODE) * 32, 1)
    rvq_encode_kernel(const __grid_constant__ RvqEncodeParams p)
{
    rvq_encode_body<BITS, MODE, SGN>(p, blockIdx.x, gridDim.x);
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
// buffer (128 columns).  Rows with a value inside the guard band go to the
// warp's exact recompute (rvq_fixup_row) while the stage is still held.
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
constexpr int TE_THREADS = 32 * (2 + 4 * TE_G);
constexpr int TE_HALF = TE_M * 128;           // a 64-coordinate half of a tile (16 KB)
constexpr int TE_TILE = 2 * TE_HALF;          // 32 KB
constexpr int TE_BOP = 2 * 128 * 128;         // B = H128 diag(s), fp16, 32 KB
__host__ __device__ constexpr int te_stages(int mode) { return mode == MODE_PAIR ? 3 : 4; }
__host__ __device__ constexpr int te_smem(int mode)
{
    return 1024 + TE_BOP + (mode == MODE_PAIR ? P4_TAB_BYTES : 0) + te_stages(mode) * TE_TILE + 256;
}
static_assert(te_smem(MODE_PAIR) <= SMEM_MAX && te_smem(MODE_SYM) <= SMEM_MAX, "tensor-memory encoder shared memory");

template <int MODE>
__global__ void __launch_bounds__(TE_THREADS, 1) rvq_encode_tc_kernel(const __grid_constant__ RvqEncodeParams p)
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
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ntiles = (p.N + TE_M - 1) / TE_M;

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
        fence_mbar_init();
    }
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
    if constexpr (MODE == MODE_PAIR)
        for (int i = threadIdx.x; i < PT_CELLS * P4_REP; i += blockDim.x) ptab[i] = p.pt.ent[i / P4_REP];
    fence_proxy_async_smem();  // B is read by the MMAs (async proxy)
    if (warp == 1) tmem_alloc(tslot, 512);
    qt_fence_before();
    __syncthreads();
    qt_fence_after();
    const uint32_t tmem = *tslot;

    if (warp == 0) {
        // ---- producer
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            int i = 0;
            for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++i) {
                const int s = i % NST;
                if (i >= NST && !mbar_wait_bounded(&x_empty[s], (uint32_t)((i / NST) - 1) & 1u)) {
                    atomicOr(&g_rvq_err, (unsigned)VQ_DEVERR_WAIT_TIMEOUT);
                    *abort_flag = 1u;
                    break;
                }
                if (*abort_flag) break;
                unsigned char *dst = ring + s * TE_TILE;
                mbar_arrive_expect_tx(&x_full[s], (uint32_t)TE_TILE);
                tma_load_2d(dst, &p.tmap, 0, t * TE_M, &x_full[s], pol);
                tma_load_2d(dst + TE_HALF, &p.tmap, 64, t * TE_M, &x_full[s], pol);
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
            for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++i) {
                const int s = i % NST, a = i % TE_G;
                bool ok = mbar_wait_bounded(&x_full[s], (uint32_t)(i / NST) & 1u);
                if (ok && i >= TE_G) ok = mbar_wait_bounded(&acc_empty[a], (uint32_t)((i / TE_G) - 1) & 1u);
                if (!ok || *abort_flag) {
                    if (!ok) atomicOr(&g_rvq_err, (unsigned)VQ_DEVERR_WAIT_TIMEOUT);
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
    } else {
        // ---- epilogue group g: tiles i with i % TE_G == g; thread = row
        const int g = (warp - 2) >> 2;
        const int q = warp & 3;  // tensor-memory lane quadrant of this warp
        const int r = 32 * q + lane;
        const uint32_t tl = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(g * 128);
        // exact-recompute tables (shuffle) and book constants
        const float tb1 = p.t1.bnd[lane];
        const int tc1 = p.t1.code[lane];
        const float tb2 = p.t2.bnd[lane];
        const int tc2 = p.t2.code[lane];
        const float tcen = p.c1[lane & ((1 << BITS) - 1)];
        [[maybe_unused]] const float b1u = p.b1[2], b2u = p.b2[2];
        [[maybe_unused]] const float bc2u = p.b1[2] - p.c1[2], dcu = p.c1[3] - p.c1[2];
        [[maybe_unused]] const float kb1 = __fdiv_rn(2.0f, b1u), kb2 = __fdiv_rn(2.0f, b2u);
        [[maybe_unused]] const float pa = p.pt.a, pbc = p.pt.bc;
        [[maybe_unused]] const uint32_t tab =
            smem_u32(ptab) + 8u * (uint32_t)(lane & (P4_REP - 1)) - (0x4B400000u << 7);
        const bool dense = p.dst_off == nullptr && p.S_dst == p.S && p.S_q == p.S;
        int i = 0;
        for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++i) {
            if (i % TE_G != g) continue;
            const int s = i % NST;
            const bool ok = mbar_wait_bounded(&acc_full[g], (uint32_t)(i / TE_G) & 1u);
            if (!__all_sync(FULL_MASK, ok) || *abort_flag) {
                if (!ok && lane == 0) atomicOr(&g_rvq_err, (unsigned)VQ_DEVERR_WAIT_TIMEOUT);
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

            flag = flag && valid;
            if (okrow && !flag) p.norms[drow] = n;
            __syncwarp();  // the fast words of a flagged row are written before its exact ones
            // rows inside the guard band: exact recompute by the warp, the row
            // read again from global memory
            unsigned fl = __ballot_sync(FULL_MASK, flag);
            while (fl) {
                const int bit = __ffs(fl) - 1;
                fl &= fl - 1;
                rvq_fixup_row<BITS, MODE == MODE_PAIR, 0>(p, nullptr, 32 * q + bit, t * TE_M + 32 * q + bit, lane, tb1, tc1,
                                                          tb2, tc2, tcen);
            }
            __syncwarp();
        }
    }

    qt_fence_before();
    __syncthreads();
    qt_fence_after();
    if (warp == 1) tmem_free(tmem, 512);
}

// ---------------------------------------------------------------- decode
//
// x_hat = n * H (c1[i1] + c2[i2]) / sqrt(D), two threads per row: lane l
// works on row l & 15 of a 16-row block and on the coordinates
// [64h, 64h + 64), h = l >> 4.  With H = [[H64, H64], [H64, -H64]], thread h
// transforms its own half, A_h = H64 u_h, scales it, swaps it with its
// partner (lane l ^ 16) and keeps A_0 + A_1 (h = 0) or A_0 - A_1 (h = 1): the
// coordinates it outputs.  The packed words of a 16-row block (contiguous in
// both streams) arrive by two bulk copies into a 3-stage ring.  For b <= 2
// the two codes of a coordinate index one merged table c1[i1] + c2[i2] (16 or
// 4 fp32 entries held one per lane and replicated across the warp, read by
// shuffle): the words of both streams are first interleaved so that a plain
// shift leaves the merged index in the low bits.  For b = 4 each stage has its
// own 16-entry table.  The fp16 half rows are staged in shared memory and
// written out coalesced.
constexpr int DEC_STAGES = 3;
constexpr int DEC_WARPS = 16;
constexpr int DROWS = 16;
__host__ __device__ constexpr int dec_stage(int bits) { return 2 * DROWS * (D * bits / 32) * 4; }
__host__ __device__ constexpr int dec_warp_bytes(int bits) { return DEC_STAGES * dec_stage(bits) + DROWS * ROW_STRIDE; }
__host__ __device__ constexpr int dec_table_bytes(int bits) { return bits == 4 ? 256 * 32 * 4 : 0; }
__host__ __device__ constexpr int dec_smem(int bits)
{
    // 1024-byte alignment of the (swizzled) stages, the b = 4 table, every
    // warp's stages, every warp's output staging, the mbarriers and the sign
    // masks of the randomised rotation (64 pair words)
    return 1024 + dec_table_bytes(bits) + DEC_WARPS * dec_warp_bytes(bits) + DEC_WARPS * DEC_STAGES * 8 + 256;
}

// Decoded values c1[i1] + c2[i2] of the 64 coordinates of one half row, as 32
// pairs (u[2k], u[2k + 1]).  w1 / w2: the half row's words of each stream.
// The two codes of a coordinate index one merged table: for b <= 2 a 16- or
// 4-entry table held one entry per lane (replicated across the warp) and read
// by shuffle; for b = 4 a 256-entry table in shared memory, replicated per
// lane (entry e of lane l at e * 32 + l, so every read is conflict-free).  The
// words of both streams are first interleaved so that a shift (b <= 2) or a
// byte extraction (b = 4) leaves the merged index i1 | i2 << b.
template <int BITS>
__device__ __forceinline__ void dec_lookup(const uint32_t (&w1)[BITS * 2], const uint32_t (&w2)[BITS * 2],
                                           float tab, const float *stab, float2 (&v)[32])
{
    constexpr int E = 32 / BITS;
    float u[64];
    if constexpr (BITS == 4) {
#pragma unroll
        for (int j = 0; j < 2 * BITS; ++j) {
            const uint32_t me = (w1[j] & 0x0F0F0F0Fu) | ((w2[j] << 4) & 0xF0F0F0F0u);
            const uint32_t mo = ((w1[j] >> 4) & 0x0F0F0F0Fu) | (w2[j] & 0xF0F0F0F0u);
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                u[j * E + 2 * m] = stab[__byte_perm(me, 0u, 0x4440u + m) * 32];
                u[j * E + 2 * m + 1] = stab[__byte_perm(mo, 0u, 0x4440u + m) * 32];
            }
        }
    } else {
        constexpr uint32_t CM = BITS == 2 ? 0x33333333u : 0x55555555u;
#pragma unroll
        for (int j = 0; j < 2 * BITS; ++j) {
            const uint32_t me = (w1[j] & CM) | ((w2[j] << BITS) & ~CM);
            const uint32_t mo = ((w1[j] >> BITS) & CM) | (w2[j] & ~CM);
#pragma unroll
            for (int m = 0; m < E / 2; ++m) {
                u[j * E + 2 * m] = __shfl_sync(FULL_MASK, tab, (int)(me >> (2 * BITS * m)));
                u[j * E + 2 * m + 1] = __shfl_sync(FULL_MASK, tab, (int)(mo >> (2 * BITS * m)));
            }
        }
    }
#pragma unroll
    for (int k = 0; k < 32; ++k) v[k] = make_float2(u[2 * k], u[2 * k + 1]);
}

template <int BITS, bool SGN>
__global__ void __launch_bounds__(DEC_WARPS * 32, 1) rvq_decode_kernel(const __grid_constant__ RvqDecodeParams p)
{
    constexpr int L = 1 << BITS;
    constexpr int W = D * BITS / 32;
    constexpr int WH = W / 2;  // words per half row
    constexpr int STG = dec_stage(BITS);
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int rr = lane & 15, hh = lane >> 4;
    unsigned char *smem = smem_1k(smem_raw);
    float *stab = reinterpret_cast<float *>(smem);  // b = 4: merged table, replicated per lane
    unsigned char *stages = smem + dec_table_bytes(BITS);  // every warp's stages, 1024-byte aligned
    unsigned char *wbuf = stages + warp * DEC_STAGES * STG;
    unsigned char *obufs = stages + DEC_WARPS * DEC_STAGES * STG;
    unsigned char *obuf = obufs + warp * DROWS * ROW_STRIDE;
    uint64_t *bars_all = reinterpret_cast<uint64_t *>(obufs + DEC_WARPS * DROWS * ROW_STRIDE);
    uint64_t *bars = bars_all + warp * DEC_STAGES;
    // sign masks: word hh * 32 + k flips output coordinates 64 hh + 2k, 64 hh + 2k + 1
    uint32_t *sgm = reinterpret_cast<uint32_t *>(bars_all + DEC_WARPS * DEC_STAGES);
    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < DEC_STAGES; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    if constexpr (BITS == 4) {
        for (int i = threadIdx.x; i < 256 * 32; i += blockDim.x) {
            const int e = i >> 5;
            stab[i] = p.c1[e & 15] + p.c2[e >> 4];
        }
    }
    if (threadIdx.x < 64) sgm[threadIdx.x] = half2_sign_mask(sign_pair(p.sgn, 2 * threadIdx.x));
    __syncthreads();
    __syncwarp();
    const uint64_t pol = l2_policy_evict_first();
    // tables: per-stage (replicated every 2^BITS lanes) and merged (index
    // i1 | i2 << BITS, replicated every 2^(2 BITS) lanes; b <= 2 only)
    const float tab = BITS == 4 ? 0.0f : p.c1[lane & (L - 1)] + p.c2[(lane >> BITS) & (L - 1)];
    const int nblk = (p.N + DROWS - 1) / DROWS;
    const int gw = blockIdx.x * DEC_WARPS + warp;
    const int tw = gridDim.x * DEC_WARPS;
    const float2 neg1 = make_float2(-1.0f, -1.0f);
    const float2 sgn = hh ? neg1 : make_float2(1.0f, 1.0f);

    auto issue = [&](int blk, int s) {
        if (lane == 0) {
            const int r0 = blk * DROWS;
            if constexpr (BITS >= 2) {
                // 16-row boxes of both streams with the 32- (b = 2) or 64-byte
                // (b = 4) swizzle; rows past N arrive as zeros
                mbar_arrive_expect_tx(&bars[s], (uint32_t)(2 * DROWS * W * 4));
                tma_load_2d(wbuf + s * STG, &p.tm1, 0, r0, &bars[s], pol);
                tma_load_2d(wbuf + s * STG + STG / 2, &p.tm2, 0, r0, &bars[s], pol);
            } else {
                const uint32_t bytes = (uint32_t)(min(DROWS, p.N - r0) * W * 4);
                mbar_arrive_expect_tx(&bars[s], 2 * bytes);
                bulk_g2s(wbuf + s * STG, p.p1 + (size_t)r0 * W, bytes, &bars[s], pol);
                bulk_g2s(wbuf + s * STG + STG / 2, p.p2 + (size_t)r0 * W, bytes, &bars[s], pol);
            }
        }
    };
#pragma unroll
    for (int s = 0; s < DEC_STAGES; ++s) {
        const int blk = gw + s * tw;
        if (blk < nblk) issue(blk, s);
    }
    for (int it = 0;; ++it) {
        const int blk = gw + it * tw;
        if (blk >= nblk) break;
        const int s = it % DEC_STAGES;
        const int row = blk * DROWS + rr;
        const bool valid = row < p.N;
        const float n = valid ? __ldg(p.norms + row) : 0.0f;
        const bool ok = mbar_wait_bounded(&bars[s], (uint32_t)(it / DEC_STAGES) & 1u);
        if (!__all_sync(FULL_MASK, ok)) {
            if (lane == 0) atomicOr(&g_rvq_err, (unsigned)VQ_DEVERR_WAIT_TIMEOUT);
            for (int k = 1; k < DEC_STAGES; ++k) {
                const int it2 = it + k;
                if (gw + it2 * tw < nblk)
                    (void)mbar_wait_bounded(&bars[it2 % DEC_STAGES], (uint32_t)(it2 / DEC_STAGES) & 1u);
            }
            return;
        }
        uint32_t w1[WH], w2[WH];
        if constexpr (BITS >= 2) {
            // 16-byte chunk k of row rr sits at chunk k ^ ((rr >> 1) & 3) (64-byte
            // rows, 64-byte swizzle) or k ^ ((rr >> 2) & 1) (32-byte rows, 32-byte
            // swizzle): the lanes of a quarter warp read distinct banks
            const unsigned char *ra = wbuf + s * STG + rr * (W * 4);
            const unsigned char *rb = ra + STG / 2;
#pragma unroll
            for (int k2 = 0; k2 < WH / 4; ++k2) {
                const int k = hh * (WH / 4) + k2;
                const int pk = BITS == 4 ? (k ^ ((rr >> 1) & 3)) : (k ^ ((rr >> 2) & 1));
                const uint4 a = *reinterpret_cast<const uint4 *>(ra + (pk << 4));
                const uint4 b = *reinterpret_cast<const uint4 *>(rb + (pk << 4));
                w1[4 * k2] = a.x; w1[4 * k2 + 1] = a.y; w1[4 * k2 + 2] = a.z; w1[4 * k2 + 3] = a.w;
                w2[4 * k2] = b.x; w2[4 * k2 + 1] = b.y; w2[4 * k2 + 2] = b.z; w2[4 * k2 + 3] = b.w;
            }
        } else {
            const uint32_t *sa = reinterpret_cast<const uint32_t *>(wbuf + s * STG) + rr * W + hh * WH;
            const uint32_t *sb = reinterpret_cast<const uint32_t *>(wbuf + s * STG + STG / 2) + rr * W + hh * WH;
#pragma unroll
            for (int i = 0; i < WH; i += 2) {
                const uint2 a = *reinterpret_cast<const uint2 *>(sa + i);
                const uint2 b = *reinterpret_cast<const uint2 *>(sb + i);
                w1[i] = a.x; w1[i + 1] = a.y;
                w2[i] = b.x; w2[i + 1] = b.y;
            }
        }
        // the words are in registers: recycle the stage
        __syncwarp();
        fence_proxy_async_smem();
        {
            const int nb = blk + DEC_STAGES * tw;
            if (nb < nblk) issue(nb, s);
        }
        float2 v[32];
        dec_lookup<BITS>(w1, w2, tab, stab + lane, v);
        // H64 on the half: coordinate bits 1-5 across the array, bit 0 in the pair
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
        // scale by n / sqrt(D), swap halves with the partner, last stage
        const float sc = __fdiv_rn(n, SQRT_D_HI);
        const float2 sc2 = make_float2(sc, sc);
        uint32_t o[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) {
            const float2 a = __fmul2_rn(make_float2(v[k].x + v[k].y, v[k].x - v[k].y), sc2);
            const float2 b = make_float2(__shfl_xor_sync(FULL_MASK, a.x, 16), __shfl_xor_sync(FULL_MASK, a.y, 16));
            // h = 0: a + b; h = 1: b - a (own half is the second operand)
            const float2 x2 = __ffma2_rn(a, sgn, b);
            const __half2 hx = __floats2half2_rn(x2.x, x2.y);
            o[k] = *reinterpret_cast<const uint32_t *>(&hx);
        }
        // o[k] holds coordinates 2k, 2k + 1 of the half; randomised signs:
        // x_hat -> diag(s) x_hat on the fp16 bits
        if constexpr (SGN) {
            const uint4 *m4 = reinterpret_cast<const uint4 *>(sgm + hh * 32);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint4 m = m4[c];
                o[4 * c] ^= m.x;
                o[4 * c + 1] ^= m.y;
                o[4 * c + 2] ^= m.z;
                o[4 * c + 3] ^= m.w;
            }
        }
        uint4 *orow = reinterpret_cast<uint4 *>(obuf + rr * ROW_STRIDE + hh * 128);
#pragma unroll
        for (int c = 0; c < 8; ++c) orow[c] = make_uint4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
        __syncwarp();
        // coalesced write-out: chunk idx = i*32 + lane is 16-byte chunk idx % 16 of row idx / 16
        const int nrows = min(DROWS, p.N - blk * DROWS);
        uint4 *gout = reinterpret_cast<uint4 *>(static_cast<__half *>(p.out) + (size_t)blk * DROWS * D);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int idx = i * 32 + lane;
            const int r = idx >> 4, c = idx & 15;
            if (r < nrows) gout[idx] = *reinterpret_cast<const uint4 *>(obuf + r * ROW_STRIDE + c * 16);
        }
        __syncwarp();
    }
}

template <int BITS, int MODE>
cudaError_t launch_enc(const RvqEncodeParams &p0, cudaStream_t stream)
{
    RvqEncodeParams p = p0;
    if (!prepare_rvq_encode(p)) return cudaErrorInvalidValue;
    auto kern = p.has_sgn ? rvq_encode_kernel<BITS, MODE, true> : rvq_encode_kernel<BITS, MODE, false>;
    constexpr int smem = enc_smem(BITS, MODE);
    constexpr int warps = enc_warps(BITS, MODE);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int nblk = (p.N + ER - 1) / ER;
    int grid = (nblk + warps - 1) / warps;
    const int sms = sm_count();
    if (grid > sms) grid = sms;
    if (grid < 1) grid = 1;
    kern<<<grid, warps * 32, smem, stream>>>(p);
    return cudaGetLastError();
}

// Launch of the tensor-memory encoder (128-row tiles): one persistent CTA per SM.
template <int MODE>
cudaError_t launch_enc_tm(const RvqEncodeParams &p0, cudaStream_t stream)
{
    RvqEncodeParams p = p0;
    p.divS = make_fastdiv((uint32_t)p.S);
    p.divH = make_fastdiv((uint32_t)p.H);
    {
        const uint64_t dims[2] = {(uint64_t)D, (uint64_t)p.N};
        const uint64_t strides[1] = {(uint64_t)D * 2};
        const uint32_t box[2] = {64u, (uint32_t)TE_M};
        if (!encode_tmap_f16(&p.tmap, p.x, 2, dims, strides, box, true, true)) return cudaErrorInvalidValue;
    }
    auto kern = rvq_encode_tc_kernel<MODE>;
    constexpr int smem = te_smem(MODE);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int ntiles = (p.N + TE_M - 1) / TE_M;
    const int grid = ntiles < sm_count() ? ntiles : sm_count();
    kern<<<grid, TE_THREADS, smem, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_enc_sym2(const RvqEncodeParams &p, cudaStream_t stream)
{
    return launch_enc_tm<MODE_SYM>(p, stream);
}


cudaError_t launch_enc_pair4(const RvqEncodeParams &p, cudaStream_t stream)
{
    return launch_enc_tm<MODE_PAIR>(p, stream);
}

template <int BITS>
cudaError_t launch_dec(const RvqDecodeParams &p0, cudaStream_t stream)
{
    RvqDecodeParams p = p0;
    if constexpr (BITS >= 2) {
        constexpr uint32_t W = D * BITS / 32;
        if (!encode_tmap_words(&p.tm1, p.p1, (uint64_t)p.N, W, DROWS, (int)(W * 4)) ||
            !encode_tmap_words(&p.tm2, p.p2, (uint64_t)p.N, W, DROWS, (int)(W * 4)))
            return cudaErrorInvalidValue;
    }
    auto kern = p.has_sgn ? rvq_decode_kernel<BITS, true> : rvq_decode_kernel<BITS, false>;
    constexpr int smem = dec_smem(BITS);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int nblk = (p.N + DROWS - 1) / DROWS;
    int grid = (nblk + DEC_WARPS - 1) / DEC_WARPS;
    const int sms = sm_count();
    if (grid > sms) grid = sms;
    if (grid < 1) grid = 1;
    kern<<<grid, DEC_WARPS * 32, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

bool prepare_rvq_encode(RvqEncodeParams &p)
{
    p.divS = make_fastdiv((uint32_t)p.S);
    p.divH = make_fastdiv((uint32_t)p.H);
    const uint64_t dims[2] = {(uint64_t)D, (uint64_t)p.N};
    const uint64_t strides[1] = {(uint64_t)D * 2};
    const uint32_t box[2] = {64u, (uint32_t)ER};
    return encode_tmap_f16(&p.tmap, p.x, 2, dims, strides, box, true, true);
}

cudaError_t launch_rvq_encode(const RvqEncodeParams &p, int bits, int mode, cudaStream_t stream)
{
    if (p.N <= 0) return cudaSuccess;
    switch (bits * 4 + mode) {
    case 1 * 4 + MODE_PLAIN: return launch_enc<1, MODE_PLAIN>(p, stream);
    case 1 * 4 + MODE_GRID: return launch_enc<1, MODE_GRID>(p, stream);
    case 1 * 4 + MODE_SYM: return launch_enc<1, MODE_SYM>(p, stream);
    case 2 * 4 + MODE_PLAIN: return launch_enc<2, MODE_PLAIN>(p, stream);
    case 2 * 4 + MODE_GRID: return launch_enc<2, MODE_GRID>(p, stream);
    case 2 * 4 + MODE_SYM: return launch_enc_sym2(p, stream);
    case 4 * 4 + MODE_PLAIN: return launch_enc<4, MODE_PLAIN>(p, stream);
    case 4 * 4 + MODE_GRID: return launch_enc<4, MODE_GRID>(p, stream);
    case 4 * 4 + MODE_PAIR: return launch_enc_pair4(p, stream);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_rvq_decode(const RvqDecodeParams &p, int bits, cudaStream_t stream)
{
    if (p.N <= 0) return cudaSuccess;
    switch (bits) {
    case 1: return launch_dec<1>(p, stream);
    case 2: return launch_dec<2>(p, stream);
    case 4: return launch_dec<4>(p, stream);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t rvq_take_device_error(unsigned *bits, cudaStream_t stream)
{
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(bits, g_rvq_err, sizeof(unsigned), 0,
                                              cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    if (*bits) e = cudaMemcpyToSymbolAsync(g_rvq_err, &zero, sizeof(unsigned), 0,
                                           cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return e;
    return cudaStreamSynchronize(stream);
}

}  // namespace vq
