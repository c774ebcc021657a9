// qjl.cu - QJL encode (sm_103a): 1-bit Johnson-Lindenstrauss sign sketches of
// keys and their norms.
//
// Method (VeloxQuant-MLX blog, tag "turboquant", "Kernel 4: QJL Encode -
// Simdgroup Sign Packing"): for each key x (D = 128 fp16 values) the m bits
// of sign(S x), a bit being 1 when the dot product with sketch row j is >= 0,
// packed least-significant bit first (bit j of 32-bit word w is row 32 w + j,
// which is the page's byte order on a little-endian machine), and ||x|| as
// fp16.
//
// Design.  The sketch is a dense product X S^T: [keys x 128] by [128 x m], on
// the tensor cores as 16 x 8 x 16 tiles (mma.sync, fp16 operands - every
// product of two fp16 values is exact - fp32 accumulation).  Persistent CTAs
// of 8 warps; the CTA copies S into shared memory once (rows padded to 272
// bytes so that ldmatrix reads are conflict-free); each warp streams its own
// 16-key blocks (two 64-coordinate TMA boxes with the 128-byte swizzle,
// double-buffered), loads the block's A fragments once (ldmatrix) and reuses
// them for every 32-column chunk of the sketch; the squared norms come from
// the same registers by paired fp32 FMAs (the squares are exact).  The signs
// of a chunk's accumulators are gathered by warp ballots and interleaved into
// one word per key.
#include <cuda_fp16.h>

#include "device_common.cuh"
#include "launch.h"

namespace vq {

namespace {

VQ_DEFINE_ERROR_WORD(g_qjl_err);

constexpr int D = 128;
constexpr int QJ_WARPS = 8;
constexpr int QJ_ROWS = 16;                 // keys per warp block
constexpr int QJ_BOX = QJ_ROWS * 128;       // one 64-coordinate box (bytes)
constexpr int QJ_STAGE = 2 * QJ_BOX;        // a block: two boxes (4 KB, 1024-aligned)
constexpr int QJ_STAGES = 2;
constexpr int SROW = D * 2 + 16;            // padded sketch row (bytes)

constexpr int qj_smem(int m)
{
    return 1024 + QJ_WARPS * QJ_STAGES * QJ_STAGE + m * SROW + QJ_WARPS * QJ_STAGES * 8;
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
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

// The 4 bits of n at the even positions of a byte.
__device__ __forceinline__ uint32_t spread4(uint32_t n)
{
    n = (n | (n << 2)) & 0x33u;
    return (n | (n << 1)) & 0x55u;
}

// W = m / 32 sign words per key; up to 4 words (16 n-tiles, 16 independent
// accumulator chains) are accumulated together.
template <int W>
__global__ void __launch_bounds__(QJ_WARPS * 32) qjl_encode_kernel(const __grid_constant__ QjlEncodeParams p)
{
    constexpr int WG = W < 4 ? W : 4;  // words per pass
    extern __shared__ __align__(128) unsigned char smem_raw[];
    unsigned char *stages = smem_1k(smem_raw);
    unsigned char *ss = stages + QJ_WARPS * QJ_STAGES * QJ_STAGE;  // sketch rows [m][SROW]
    uint64_t *bars = reinterpret_cast<uint64_t *>(ss + p.m * SROW);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nblk = (p.N + QJ_ROWS - 1) / QJ_ROWS;
    const int tw = gridDim.x * QJ_WARPS;      // warps of the grid
    const int gw = blockIdx.x * QJ_WARPS + warp;

    unsigned char *my_st = stages + warp * QJ_STAGES * QJ_STAGE;
    uint64_t *my_bar = bars + warp * QJ_STAGES;
    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < QJ_STAGES; ++s) mbar_init(&my_bar[s], 1);
        fence_mbar_init();
    }
    __syncwarp();
    const uint64_t pol = l2_policy_evict_first();
    auto issue = [&](int blk, int st) {
        if (lane == 0) {
            unsigned char *dst = my_st + st * QJ_STAGE;
            mbar_arrive_expect_tx(&my_bar[st], (uint32_t)QJ_STAGE);
            tma_load_2d(dst, &p.tmx, 0, blk * QJ_ROWS, &my_bar[st], pol);
            tma_load_2d(dst + QJ_BOX, &p.tmx, 64, blk * QJ_ROWS, &my_bar[st], pol);
        }
    };
#pragma unroll
    for (int s = 0; s < QJ_STAGES; ++s)
        if (gw + s * tw < nblk) issue(gw + s * tw, s);

    // the sketch, once per CTA: 16-byte pieces into padded rows
    {
        const uint4 *src = static_cast<const uint4 *>(p.s);
        for (int i = threadIdx.x; i < p.m * (D / 8); i += blockDim.x) {
            const int r = i >> 4, c = i & 15;
            *reinterpret_cast<uint4 *>(ss + r * SROW + c * 16) = __ldg(src + i);
        }
    }
    __syncthreads();

    const int g8 = lane >> 2, t4 = lane & 3;
    const uint32_t sbase = smem_u32(ss);
    // ldmatrix rows: A (keys) row (lane & 7) + 8 ((lane >> 3) & 1), 16-byte
    // chunk 2 kt' + (lane >> 4) of its box; B (sketch rows) for two n-tiles:
    // row (lane & 7) + 8 (lane >> 4), chunk 2 kt + ((lane >> 3) & 1)
    const int arow = (lane & 7) + 8 * ((lane >> 3) & 1), ach = lane >> 4;
    const int brow = (lane & 7) + 8 * (lane >> 4), bch = (lane >> 3) & 1;

    for (int it = 0;; ++it) {
        const int blk = gw + it * tw;
        if (blk >= nblk) break;
        const int st = it % QJ_STAGES;
        const bool ok = mbar_wait_bounded(&my_bar[st], (uint32_t)(it / QJ_STAGES) & 1u);
        if (!__all_sync(FULL_MASK, ok)) {
            if (lane == 0) atomicOr(&g_qjl_err, (unsigned)VQ_DEVERR_WAIT_TIMEOUT);
            for (int k = 1; k < QJ_STAGES; ++k) {
                const int it2 = it + k;
                if (gw + it2 * tw < nblk)
                    (void)mbar_wait_bounded(&my_bar[it2 % QJ_STAGES], (uint32_t)(it2 / QJ_STAGES) & 1u);
            }
            break;
        }
        const uint32_t xb = smem_u32(my_st + st * QJ_STAGE);
        uint32_t a[8][4];
#pragma unroll
        for (int kt = 0; kt < 8; ++kt)
            ldsm_x4(xb + (kt >> 2) * QJ_BOX + swz128(arow, 2 * (kt & 3) + ach), a[kt][0], a[kt][1], a[kt][2],
                    a[kt][3]);
        // the stage is consumed (the fragments are in registers): refill it
        __syncwarp();
        fence_proxy_async_smem();
        if (blk + QJ_STAGES * tw < nblk) issue(blk + QJ_STAGES * tw, st);

        const int row0 = blk * QJ_ROWS;
        // squared norms from the fragments in registers (the tensor pipe is
        // the busy one): keys g8 (registers 0, 2) and g8 + 8 (1, 3), 32 exact
        // squares each per lane in paired fp32 FMAs, then the 4 lanes of a key
        {
            float2 qa = make_float2(0.0f, 0.0f), qb = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int kt = 0; kt < 8; ++kt) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&a[kt][j]));
                    if (j & 1) qb = __ffma2_rn(f, f, qb);
                    else qa = __ffma2_rn(f, f, qa);
                }
            }
            float sa = qa.x + qa.y, sb = qb.x + qb.y;
            sa += __shfl_xor_sync(FULL_MASK, sa, 1);
            sb += __shfl_xor_sync(FULL_MASK, sb, 1);
            sa += __shfl_xor_sync(FULL_MASK, sa, 2);
            sb += __shfl_xor_sync(FULL_MASK, sb, 2);
            if (t4 == 0) {
                __half *nr = static_cast<__half *>(p.norms);
                if (row0 + g8 < p.N) nr[row0 + g8] = __float2half_rn(__fsqrt_rn(sa));
                if (row0 + g8 + 8 < p.N) nr[row0 + g8 + 8] = __float2half_rn(__fsqrt_rn(sb));
            }
        }
        // signs, WG words (32 sketch rows each) per pass
#pragma unroll
        for (int w0 = 0; w0 < W; w0 += WG) {
            float acc[4 * WG][4];
#pragma unroll
            for (int nt = 0; nt < 4 * WG; ++nt)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[nt][j] = 0.0f;
#pragma unroll
            for (int kt = 0; kt < 8; ++kt) {
#pragma unroll
                for (int np = 0; np < 2 * WG; ++np) {  // a pair of n-tiles per ldmatrix
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(sbase + (uint32_t)((32 * w0 + 16 * np + brow) * SROW + (2 * kt + bch) * 16), b0, b1,
                            b2, b3);
                    // b0, b1: sketch rows 0..7 of the pair (k 0..7, 8..15); b2, b3: rows 8..15
                    mma_16816(acc[2 * np], a[kt][0], a[kt][1], a[kt][2], a[kt][3], b0, b1);
                    mma_16816(acc[2 * np + 1], a[kt][0], a[kt][1], a[kt][2], a[kt][3], b2, b3);
                }
            }
            // lane 4 g8 + t4 holds keys g8 and g8 + 8 at sketch columns 2 t4,
            // 2 t4 + 1 of each n-tile; nibble r of a ballot is key r's four
            // even (or odd) columns of that n-tile
            const int r = lane & 15;
            const int sh = 4 * (r & 7);
#pragma unroll
            for (int w = 0; w < WG; ++w) {
                uint32_t word = 0;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int nt = 4 * w + q;
                    const uint32_t e0 = __ballot_sync(FULL_MASK, acc[nt][0] >= 0.0f);
                    const uint32_t o0 = __ballot_sync(FULL_MASK, acc[nt][1] >= 0.0f);
                    const uint32_t e1 = __ballot_sync(FULL_MASK, acc[nt][2] >= 0.0f);
                    const uint32_t o1 = __ballot_sync(FULL_MASK, acc[nt][3] >= 0.0f);
                    const uint32_t ev = r < 8 ? e0 : e1, od = r < 8 ? o0 : o1;
                    const uint32_t byte = spread4((ev >> sh) & 15u) | (spread4((od >> sh) & 15u) << 1);
                    word |= byte << (8 * q);
                }
                if (lane < 16 && row0 + r < p.N) p.packed[(size_t)(row0 + r) * W + w0 + w] = word;
            }
        }
    }
}

}  // namespace

cudaError_t launch_qjl_encode(const QjlEncodeParams &p0, cudaStream_t stream)
{
    if (p0.N <= 0) return cudaSuccess;
    QjlEncodeParams p = p0;
    {
        const uint64_t dims[2] = {(uint64_t)D, (uint64_t)p.N};
        const uint64_t strides[1] = {(uint64_t)D * 2};
        const uint32_t box[2] = {64u, (uint32_t)QJ_ROWS};
        if (!encode_tmap_f16(&p.tmx, p.x, 2, dims, strides, box, true, true)) return cudaErrorInvalidValue;
    }
    const int smem = qj_smem(p.m);
    void (*kern)(QjlEncodeParams) = nullptr;
    switch (p.m / 32) {
    case 1: kern = qjl_encode_kernel<1>; break;
    case 2: kern = qjl_encode_kernel<2>; break;
    case 3: kern = qjl_encode_kernel<3>; break;
    case 4: kern = qjl_encode_kernel<4>; break;
    case 5: kern = qjl_encode_kernel<5>; break;
    case 6: kern = qjl_encode_kernel<6>; break;
    case 7: kern = qjl_encode_kernel<7>; break;
    case 8: kern = qjl_encode_kernel<8>; break;
    default: return cudaErrorInvalidValue;
    }
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, QJ_WARPS * 32, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    const int nblk = (p.N + QJ_ROWS - 1) / QJ_ROWS;
    const int want = (nblk + QJ_WARPS - 1) / QJ_WARPS;
    const int grid = want < sm_count() * per_sm ? want : sm_count() * per_sm;
    kern<<<grid, QJ_WARPS * 32, smem, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t qjl_take_device_error(unsigned *bits, cudaStream_t stream)
{
    *bits = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(bits, g_qjl_err, sizeof(unsigned), 0, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    if (*bits) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbolAsync(g_qjl_err, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice, stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    }
    return e;
}

}  // namespace vq
