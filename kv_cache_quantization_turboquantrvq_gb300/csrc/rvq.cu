// rvq.cu - TurboQuantRVQ encode+pack and unpack+dequant kernels for sm_103a.
//
// The encoders' device code (method, design and exactness notes) is in
// rvq_encode.cuh; here are their kernels (one persistent CTA per SM, each
// running the shared body over its share of the rows), the decoder and the
// launchers.
#include <cuda_fp16.h>

#include "device_common.cuh"
#include "launch.h"

#include <cstring>
#include <mutex>

namespace vq {
VQ_DEFINE_ERROR_WORD(g_rvq_err);
}  // namespace vq

#define VQ_RVQ_ERR g_rvq_err
#include "rvq_encode.cuh"

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

// The tensor-memory encoder of the library's books (rvq_encode.cuh), one
// persistent CTA per SM.
template <int MODE>
__global__ void __launch_bounds__(TE_THREADS, 1) rvq_encode_tc_kernel(const __grid_constant__ RvqEncodeParams p)
{
    rvq_encode_tm_body<MODE>(p, blockIdx.x, gridDim.x);
}

// ---------------------------------------------------------------- decode
//
// x_hat = n * H (c1[i1] + c2[i2]) / sqrt(D).  Two kernels share the table
// decode below: rvq_decode_row_kernel (b = 2, 4: a thread per row) and
// rvq_decode_kernel (b = 1: two threads per row, whose 16-byte rows are too
// narrow for the row kernel's 16-byte chunks per half row).
//
// rvq_decode_kernel: lane l works on row l & 15 of a 16-row block and on the
// coordinates [64h, 64h + 64), h = l >> 4.  With H = [[H64, H64], [H64,
// -H64]], thread h transforms its own half, A_h = H64 u_h, scales it, swaps
// it with its partner (lane l ^ 16) and keeps A_0 + A_1 (h = 0) or A_0 - A_1
// (h = 1): the coordinates it outputs.  The packed words of a 16-row block
// (contiguous in both streams) arrive by two bulk copies into a 3-stage ring.
// The fp16 half rows are staged in shared memory and written out coalesced.
constexpr int DEC_STAGES = 3;
constexpr int DEC_WARPS = 16;
constexpr int DROWS = 16;
__host__ __device__ constexpr int dec_stage(int bits) { return 2 * DROWS * (D * bits / 32) * 4; }
__host__ __device__ constexpr int dec_warp_bytes(int bits) { return DEC_STAGES * dec_stage(bits) + DROWS * ROW_STRIDE; }
// b = 4: the merged 256-entry table, replicated per lane (row kernel)
__host__ __device__ constexpr int dec_table_bytes(int bits) { return bits == 4 ? 256 * 32 * 4 : 0; }
__host__ __device__ constexpr int dec_smem(int bits)
{
    // 1024-byte alignment, every warp's stages, every warp's output staging,
    // the mbarriers, the sign masks of the randomised rotation (64 pair
    // words) and the CTA's block counter
    return 1024 + DEC_WARPS * dec_warp_bytes(bits) + DEC_WARPS * DEC_STAGES * 8 + 256 + 16;
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
    static_assert(BITS == 1, "b = 2 and b = 4 decode in rvq_decode_row_kernel");
    constexpr int L = 1 << BITS;
    constexpr int W = D * BITS / 32;
    constexpr int WH = W / 2;  // words per half row
    constexpr int STG = dec_stage(BITS);
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int rr = lane & 15, hh = lane >> 4;
    unsigned char *stages = smem_1k(smem_raw);  // every warp's stages
    unsigned char *wbuf = stages + warp * DEC_STAGES * STG;
    unsigned char *obufs = stages + DEC_WARPS * DEC_STAGES * STG;
    unsigned char *obuf = obufs + warp * DROWS * ROW_STRIDE;
    uint64_t *bars_all = reinterpret_cast<uint64_t *>(obufs + DEC_WARPS * DROWS * ROW_STRIDE);
    uint64_t *bars = bars_all + warp * DEC_STAGES;
    // sign masks: word hh * 32 + k flips output coordinates 64 hh + 2k, 64 hh + 2k + 1
    uint32_t *sgm = reinterpret_cast<uint32_t *>(bars_all + DEC_WARPS * DEC_STAGES);
    // the CTA takes the blocks [lo, hi) and its warps claim them one at a
    // time (a shared counter), so that they finish together
    uint32_t *claimed = sgm + 64;
    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < DEC_STAGES; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    if (threadIdx.x < 64) sgm[threadIdx.x] = half2_sign_mask(sign_pair(p.sgn, 2 * threadIdx.x));
    if (threadIdx.x == 0) *claimed = 0u;
    __syncthreads();
    const uint64_t pol = l2_policy_evict_first();
    // the merged table, index i1 | i2 << BITS, replicated every 2^(2 BITS) lanes
    const float tab = p.c1[lane & (L - 1)] + p.c2[(lane >> BITS) & (L - 1)];
    const int nblk = (p.N + DROWS - 1) / DROWS;
    const int lo = (int)((long long)blockIdx.x * nblk / gridDim.x);
    const int hi = (int)((long long)(blockIdx.x + 1) * nblk / gridDim.x);
    auto claim = [&]() {
        int b = 0;
        if (lane == 0) b = lo + (int)atomicAdd(claimed, 1u);
        return __shfl_sync(FULL_MASK, b, 0);
    };
    const float2 neg1 = make_float2(-1.0f, -1.0f);
    const float2 sgn = hh ? neg1 : make_float2(1.0f, 1.0f);

    auto issue = [&](int blk, int s) {
        if (lane == 0) {
            const int r0 = blk * DROWS;
            const uint32_t bytes = (uint32_t)(min(DROWS, p.N - r0) * W * 4);
            mbar_arrive_expect_tx(&bars[s], 2 * bytes);
            bulk_g2s(wbuf + s * STG, p.p1 + (size_t)r0 * W, bytes, &bars[s], pol);
            bulk_g2s(wbuf + s * STG + STG / 2, p.p2 + (size_t)r0 * W, bytes, &bars[s], pol);
        }
    };
    // sb[s]: the block staged in stage s (claims are increasing and consumed
    // in claim order), held as three scalars
    static_assert(DEC_STAGES == 3, "three stages per warp");
    int sb0 = claim();
    if (sb0 < hi) issue(sb0, 0);
    int sb1 = claim();
    if (sb1 < hi) issue(sb1, 1);
    int sb2 = claim();
    if (sb2 < hi) issue(sb2, 2);
    for (int it = 0;; ++it) {
        const int s = it % DEC_STAGES;
        const int blk = s == 0 ? sb0 : (s == 1 ? sb1 : sb2);
        if (blk >= hi) break;
        const int row = blk * DROWS + rr;
        const bool valid = row < p.N;
        const float n = valid ? __ldg(p.norms + row) : 0.0f;
        const bool ok = mbar_wait_bounded(&bars[s], (uint32_t)(it / DEC_STAGES) & 1u);
        if (!__all_sync(FULL_MASK, ok)) {
            if (lane == 0) atomicOr(&g_rvq_err, (unsigned)VQ_DEVERR_WAIT_TIMEOUT);
            // the other stages' copies, if any, are still in flight
            for (int k = 1; k < DEC_STAGES; ++k) {
                const int it2 = it + k, s2 = it2 % DEC_STAGES;
                if ((s2 == 0 ? sb0 : (s2 == 1 ? sb1 : sb2)) < hi)
                    (void)mbar_wait_bounded(&bars[s2], (uint32_t)(it2 / DEC_STAGES) & 1u);
            }
            return;
        }
        uint32_t w1[WH], w2[WH];
        {
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
            const int nb = claim();
            if (s == 0)
                sb0 = nb;
            else if (s == 1)
                sb1 = nb;
            else
                sb2 = nb;
            if (nb < hi) issue(nb, s);
        }
        float2 v[32];
        dec_lookup<BITS>(w1, w2, tab, nullptr, v);
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
    if (!prepare_rvq_encode(p, ER)) return cudaErrorInvalidValue;
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
    if (!prepare_rvq_encode(p, TE_M)) return cudaErrorInvalidValue;
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

// Decode, b in {2, 4}, a thread per row: a lane holds all 128 coordinates
// of its row, so every Hadamard stage is register arithmetic (fp32x2
// butterflies; the last stage two adds instead of a partner exchange).
// The values c1[i1] + c2[i2] come from tables in shared memory, replicated
// per lane (entry e of lane l at 32 e + l): b = 4, the merged per-coordinate
// table (256 entries, read as 4 bytes); b = 2, a table per coordinate pair
// (2k, 2k + 1), indexed by both coordinates' merged 4-bit indices and holding
// (T[a] + T[b], T[a] - T[b]) with T[i] = c1[i & 3] + c2[i >> 2], so that the
// first stage (bit 0) is taken in the lookup, one 8-byte read per pair (8.8
// instructions per element at b = 2, against 10.4 for two threads per row).
// 32-row blocks (one row per lane) arrive as 2D TMA boxes of both streams
// (32- or 64-byte swizzle) into a 2-stage ring per warp; the fp16 rows are
// staged in shared memory (16-byte chunks swizzled by row) and written out as
// whole contiguous blocks.  12 warps per SM (168 registers a thread).
constexpr int DR_WARPS = 12;
constexpr int DR_ROWS = 32;
constexpr int DR_NST = 2;
__host__ __device__ constexpr int dr_w(int bits) { return D * bits / 32; }       // words per row and stream
__host__ __device__ constexpr int dr_stage(int bits) { return 2 * DR_ROWS * dr_w(bits) * 4; }  // both streams
constexpr int DR_OUT = DR_ROWS * 256;                   // fp16 rows of a block: 8 KB
__host__ __device__ constexpr int dr_table_bytes(int bits) { return bits == 2 ? 256 * 32 * 8 : dec_table_bytes(bits); }
__host__ __device__ constexpr int dr_smem(int bits)
{
    return 1024 + dr_table_bytes(bits) + DR_WARPS * (DR_NST * dr_stage(bits) + DR_OUT) + DR_WARPS * DR_NST * 8 + 256 + 16;
}
static_assert(dr_smem(4) <= SMEM_MAX && dr_smem(2) <= SMEM_MAX, "row decoder shared memory");

// b = 2: the decoded pairs (u[2k] + u[2k + 1], u[2k] - u[2k + 1]) of the 64
// coordinates of one half row (k = 0 .. 31), from the half row's words and
// the per-lane pair table (this lane's replica).  me / mo hold the merged
// 4-bit indices of the even / odd coordinates (nibble m of word j: coordinate
// 16 j + 2 m, resp. + 1); their nibbles are paired into bytes, byte q of A
// for pair 2q and of B for pair 2q + 1.
__device__ __forceinline__ void dec_lookup_pairs2(const uint32_t (&w1)[4], const uint32_t (&w2)[4],
                                                  const float2 *ptab, float2 (&v)[32])
{
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t me = (w1[j] & 0x33333333u) | ((w2[j] << 2) & 0xCCCCCCCCu);
        const uint32_t mo = ((w1[j] >> 2) & 0x33333333u) | (w2[j] & 0xCCCCCCCCu);
        const uint32_t a = (me & 0x0F0F0F0Fu) | ((mo << 4) & 0xF0F0F0F0u);
        const uint32_t b = ((me >> 4) & 0x0F0F0F0Fu) | (mo & 0xF0F0F0F0u);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            v[8 * j + 2 * q] = ptab[__byte_perm(a, 0u, 0x4440u + q) * 32];
            v[8 * j + 2 * q + 1] = ptab[__byte_perm(b, 0u, 0x4440u + q) * 32];
        }
    }
}

template <int BITS, bool SGN>
__global__ void __launch_bounds__(DR_WARPS * 32, 1) rvq_decode_row_kernel(const __grid_constant__ RvqDecodeParams p)
{
    constexpr int DR_W = dr_w(BITS);
    constexpr int DR_STAGE = dr_stage(BITS);
    constexpr int WH = DR_W / 2;  // words per half row
    extern __shared__ __align__(128) unsigned char smem_raw[];
    unsigned char *smem0 = smem_1k(smem_raw);
    float *stab = reinterpret_cast<float *>(smem0);    // b = 4: merged table, replicated per lane
    float2 *ptab = reinterpret_cast<float2 *>(smem0);  // b = 2: pair table, replicated per lane
    unsigned char *smem = smem0 + dr_table_bytes(BITS);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    unsigned char *wbuf = smem + warp * (DR_NST * DR_STAGE);
    unsigned char *obuf = smem + DR_WARPS * DR_NST * DR_STAGE + warp * DR_OUT;
    uint64_t *bars_all = reinterpret_cast<uint64_t *>(smem + DR_WARPS * (DR_NST * DR_STAGE + DR_OUT));
    uint64_t *bars = bars_all + warp * DR_NST;
    // sign masks: word k flips output coordinates 2k, 2k + 1
    uint32_t *sgm = reinterpret_cast<uint32_t *>(bars_all + DR_WARPS * DR_NST);
    uint32_t *claimed = sgm + 64;
    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < DR_NST; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    if (threadIdx.x < 64) sgm[threadIdx.x] = half2_sign_mask(sign_pair(p.sgn, 2 * threadIdx.x));
    if (threadIdx.x == 0) *claimed = 0u;
    if constexpr (BITS == 4) {
        // entry e (warp-uniform: 32 | blockDim) from the two books held one
        // entry per lane: no memory latency per entry
        const float t1 = p.c1[lane & 15], t2 = p.c2[lane & 15];
        for (int i = threadIdx.x; i < 256 * 32; i += blockDim.x) {
            const int e = i >> 5;
            stab[i] = __shfl_sync(FULL_MASK, t1, e & 15) + __shfl_sync(FULL_MASK, t2, e >> 4);
        }
    } else {
        // T[lane & 15], index i1 | i2 << 2; entry e (warp-uniform: 32 | blockDim)
        // pairs a = e & 15 (even coordinate) with b = e >> 4 (odd)
        const float t = p.c1[lane & 3] + p.c2[(lane >> 2) & 3];
        for (int i = threadIdx.x; i < 256 * 32; i += blockDim.x) {
            const int e = i >> 5;
            const float ta = __shfl_sync(FULL_MASK, t, e & 15), tb = __shfl_sync(FULL_MASK, t, e >> 4);
            ptab[i] = make_float2(ta + tb, ta - tb);
        }
    }
    __syncthreads();
    const uint64_t pol = l2_policy_evict_first();
    const int nblk = (p.N + DR_ROWS - 1) / DR_ROWS;
    const int lo = (int)((long long)blockIdx.x * nblk / gridDim.x);
    const int hi = (int)((long long)(blockIdx.x + 1) * nblk / gridDim.x);
    auto claim = [&]() {
        int b = 0;
        if (lane == 0) b = lo + (int)atomicAdd(claimed, 1u);
        return __shfl_sync(FULL_MASK, b, 0);
    };
    auto issue = [&](int blk, int s) {
        if (lane == 0) {
            mbar_arrive_expect_tx(&bars[s], (uint32_t)DR_STAGE);
            tma_load_2d(wbuf + s * DR_STAGE, &p.tm1, 0, blk * DR_ROWS, &bars[s], pol);
            tma_load_2d(wbuf + s * DR_STAGE + DR_STAGE / 2, &p.tm2, 0, blk * DR_ROWS, &bars[s], pol);
        }
    };
    static_assert(DR_NST == 2, "two stages per warp");
    int sb0 = claim();
    if (sb0 < hi) issue(sb0, 0);
    int sb1 = claim();
    if (sb1 < hi) issue(sb1, 1);
    const float2 neg1 = make_float2(-1.0f, -1.0f);
    for (int it = 0;; ++it) {
        const int s = it & 1;
        const int blk = s ? sb1 : sb0;
        if (blk >= hi) break;
        const int row = blk * DR_ROWS + lane;
        const bool valid = row < p.N;
        const float n = valid ? __ldg(p.norms + row) : 0.0f;
        const bool ok = mbar_wait_bounded(&bars[s], (uint32_t)(it >> 1) & 1u);
        if (!__all_sync(FULL_MASK, ok)) {
            if (lane == 0) atomicOr(&g_rvq_err, (unsigned)VQ_DEVERR_WAIT_TIMEOUT);
            const int it2 = it + 1;  // the other stage's copy, if any, is still in flight
            if ((s ? sb0 : sb1) < hi) (void)mbar_wait_bounded(&bars[it2 & 1], (uint32_t)(it2 >> 1) & 1u);
            return;
        }
        // the row's words (rows of 4 W bytes with the matching swizzle: 16-byte
        // chunk k at k ^ ((lane >> 2) & 1) for 32-byte rows, k ^ ((lane >> 1) & 3)
        // for 64-byte rows), half row h from chunks [h C, h C + C)
        constexpr int CH = DR_W / 8;  // 16-byte chunks per half row
        const unsigned char *ra = wbuf + s * DR_STAGE + lane * (DR_W * 4);
        const unsigned char *rb = ra + DR_STAGE / 2;
        auto words = [&](int h, uint32_t (&a)[WH], uint32_t (&b)[WH]) {
#pragma unroll
            for (int k2 = 0; k2 < CH; ++k2) {
                const int k = h * CH + k2;
                const int pk = BITS == 4 ? (k ^ ((lane >> 1) & 3)) : (k ^ ((lane >> 2) & 1));
                const uint4 x = *reinterpret_cast<const uint4 *>(ra + (pk << 4));
                const uint4 y = *reinterpret_cast<const uint4 *>(rb + (pk << 4));
                a[4 * k2] = x.x; a[4 * k2 + 1] = x.y; a[4 * k2 + 2] = x.z; a[4 * k2 + 3] = x.w;
                b[4 * k2] = y.x; b[4 * k2 + 1] = y.y; b[4 * k2 + 2] = y.z; b[4 * k2 + 3] = y.w;
            }
        };
        // all of the row's words into registers first, so that the stage is
        // refilled before the table decode
        uint32_t a0[WH], b0[WH], a1[WH], b1[WH];
        words(0, a0, b0);
        words(1, a1, b1);
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
        // y_hat of the two halves, H64 on each (coordinate bits 1-5 across the
        // array, bit 0 in the pair: already taken by the b = 2 pair table),
        // then bit 6 across the halves
        float2 v0[32], v1[32];
        if constexpr (BITS == 2) {
            dec_lookup_pairs2(a0, b0, ptab + lane, v0);
            dec_lookup_pairs2(a1, b1, ptab + lane, v1);
        } else {
            dec_lookup<BITS>(a0, b0, 0.0f, stab + lane, v0);
            dec_lookup<BITS>(a1, b1, 0.0f, stab + lane, v1);
        }
#pragma unroll
        for (int h = 1; h < 32; h <<= 1) {
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                if ((k & h) == 0) {
                    const float2 a0 = v0[k], b0 = v0[k + h];
                    v0[k] = __fadd2_rn(a0, b0);
                    v0[k + h] = __ffma2_rn(b0, neg1, a0);
                    const float2 a1 = v1[k], b1 = v1[k + h];
                    v1[k] = __fadd2_rn(a1, b1);
                    v1[k + h] = __ffma2_rn(b1, neg1, a1);
                }
            }
        }
        // bit 6, bit 0, the scale n / sqrt(D), fp16, signs; staged by row
        const float sc = __fdiv_rn(n, SQRT_D_HI);
        const float2 sc2 = make_float2(sc, sc);
        unsigned char *orow = obuf + lane * 256;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            uint32_t o0[4], o1[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int k = 4 * c + e;
                const float2 a = v0[k], b = v1[k];
                const float2 u = __fadd2_rn(a, b), w = __ffma2_rn(b, neg1, a);  // coordinates 2k, 2k+1 | 64 + 2k, 64 + 2k + 1 (b = 4: before bit 0)
                const float2 xu = BITS == 2 ? __fmul2_rn(u, sc2) : __fmul2_rn(make_float2(u.x + u.y, u.x - u.y), sc2);
                const float2 xw = BITS == 2 ? __fmul2_rn(w, sc2) : __fmul2_rn(make_float2(w.x + w.y, w.x - w.y), sc2);
                const __half2 hu = __floats2half2_rn(xu.x, xu.y), hw = __floats2half2_rn(xw.x, xw.y);
                o0[e] = *reinterpret_cast<const uint32_t *>(&hu);
                o1[e] = *reinterpret_cast<const uint32_t *>(&hw);
                if constexpr (SGN) {
                    o0[e] ^= sgm[k];
                    o1[e] ^= sgm[32 + k];
                }
            }
            // 16-byte chunk c (coordinates 8c .. 8c + 7) and chunk 8 + c, swizzled by row
            *reinterpret_cast<uint4 *>(orow + ((c ^ (lane & 15)) << 4)) = make_uint4(o0[0], o0[1], o0[2], o0[3]);
            *reinterpret_cast<uint4 *>(orow + (((8 + c) ^ (lane & 15)) << 4)) = make_uint4(o1[0], o1[1], o1[2], o1[3]);
        }
        __syncwarp();
        // coalesced write-out: 16-byte chunk idx = i * 32 + lane is chunk idx % 16 of row idx / 16
        const int nrows = min(DR_ROWS, p.N - blk * DR_ROWS);
        uint4 *gout = reinterpret_cast<uint4 *>(static_cast<__half *>(p.out) + (size_t)blk * DR_ROWS * D);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int idx = i * 32 + lane;
            const int r = idx >> 4, c = idx & 15;
            if (r < nrows) gout[idx] = *reinterpret_cast<const uint4 *>(obuf + r * 256 + ((c ^ (r & 15)) << 4));
        }
        __syncwarp();
    }
}

template <int BITS>
cudaError_t launch_dec(const RvqDecodeParams &p, cudaStream_t stream)
{
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

bool prepare_rvq_encode(RvqEncodeParams &p, int box_rows)
{
    p.divS = make_fastdiv((uint32_t)p.S);
    p.divH = make_fastdiv((uint32_t)p.H);
    const uint64_t dims[2] = {(uint64_t)D, (uint64_t)p.N};
    const uint64_t strides[1] = {(uint64_t)D * 2};
    const uint32_t box[2] = {64u, (uint32_t)box_rows};
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

namespace {
template <int BITS>
cudaError_t launch_dec_row(const RvqDecodeParams &p0, cudaStream_t stream)
{
    RvqDecodeParams p = p0;
    constexpr int W = dr_w(BITS);
    if (!encode_tmap_words(&p.tm1, p.p1, (uint64_t)p.N, W, DR_ROWS, W * 4) ||
        !encode_tmap_words(&p.tm2, p.p2, (uint64_t)p.N, W, DR_ROWS, W * 4))
        return cudaErrorInvalidValue;
    auto kern = p.has_sgn ? rvq_decode_row_kernel<BITS, true> : rvq_decode_row_kernel<BITS, false>;
    constexpr int smem = dr_smem(BITS);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int nblk = (p.N + DR_ROWS - 1) / DR_ROWS;
    int grid = (nblk + DR_WARPS - 1) / DR_WARPS;
    const int sms = sm_count();
    if (grid > sms) grid = sms;
    if (grid < 1) grid = 1;
    kern<<<grid, DR_WARPS * 32, smem, stream>>>(p);
    return cudaGetLastError();
}
}  // namespace

cudaError_t launch_rvq_decode(const RvqDecodeParams &p, int bits, cudaStream_t stream)
{
    if (p.N <= 0) return cudaSuccess;
    switch (bits) {
    case 1: return launch_dec<1>(p, stream);
    case 2: return launch_dec_row<2>(p, stream);
    case 4: return launch_dec_row<4>(p, stream);
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

// ------------------------------------------------ pair tables in device memory

namespace {
constexpr int kPtSlots = 16;
constexpr int kPtDevices = 8;
__device__ uint2 g_pt_slots[kPtSlots][PT_CELLS];
struct PtSlot {
    bool used = false;
    bool done = false;  // the upload is known to be complete
    uint2 ent[PT_CELLS];
    cudaEvent_t uploaded = nullptr;
};
std::mutex g_pt_mu;
PtSlot g_pt[kPtDevices][kPtSlots];
}  // namespace

const uint2 *pair_table_device(const PairTable &pt, cudaStream_t stream)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kPtDevices) return nullptr;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return nullptr;
    const bool capturing = cap != cudaStreamCaptureStatusNone;
    void *base = nullptr;
    if (cudaGetSymbolAddress(&base, g_pt_slots) != cudaSuccess) return nullptr;
    std::lock_guard<std::mutex> lock(g_pt_mu);
    for (int i = 0; i < kPtSlots; ++i) {
        PtSlot &sl = g_pt[dev][i];
        if (!sl.used || std::memcmp(sl.ent, pt.ent, sizeof(sl.ent)) != 0) continue;
        if (!sl.done) {
            // during a capture no event may be queried or waited on: use the
            // slot only once its upload is known to be complete
            if (capturing) return nullptr;
            const cudaError_t q = cudaEventQuery(sl.uploaded);
            if (q == cudaSuccess) {
                sl.done = true;
            } else if (q == cudaErrorNotReady) {
                // uploaded on another stream and not yet done: order this one after it
                if (cudaStreamWaitEvent(stream, sl.uploaded, 0) != cudaSuccess) return nullptr;
            } else {
                return nullptr;
            }
        }
        return static_cast<const uint2 *>(base) + (size_t)i * PT_CELLS;
    }
    if (capturing) return nullptr;  // no upload inside a capture
    for (int i = 0; i < kPtSlots; ++i) {
        PtSlot &sl = g_pt[dev][i];
        if (sl.used) continue;
        std::memcpy(sl.ent, pt.ent, sizeof(sl.ent));
        if (sl.uploaded == nullptr && cudaEventCreateWithFlags(&sl.uploaded, cudaEventDisableTiming) != cudaSuccess) {
            sl.uploaded = nullptr;
            return nullptr;
        }
        if (cudaMemcpyToSymbolAsync(g_pt_slots, sl.ent, sizeof(sl.ent), (size_t)i * sizeof(sl.ent),
                                    cudaMemcpyHostToDevice, stream) != cudaSuccess ||
            cudaEventRecord(sl.uploaded, stream) != cudaSuccess)
            return nullptr;
        sl.used = true;
        sl.done = false;
        return static_cast<const uint2 *>(base) + (size_t)i * PT_CELLS;
    }
    return nullptr;  // every slot taken
}

}  // namespace vq
