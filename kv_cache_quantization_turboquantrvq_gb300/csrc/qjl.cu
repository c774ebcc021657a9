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
// Design.  The sketch is the dense product X S^T: [keys x 128] by [128 x m],
// the one real contraction of the path, on the 5th-generation tensor cores
// (tcgen05.mma from shared memory into tensor memory; fp16 operands - every
// product of two fp16 values is exact - fp32 accumulation).  See the
// tcgen05 section below for the tiling and the roles of the warps.
#include <cuda_fp16.h>

#include "device_common.cuh"
#include "launch.h"
#include "tcgen05.cuh"

namespace vq {

namespace {

VQ_DEFINE_ERROR_WORD(g_qjl_err);

constexpr int D = 128;
// ------------------------------------------------------------ tcgen05 path
//
// The sketch of a tile of 128 keys is one D = X S^T of M = 128, N = m,
// K = 128 on the 5th-generation tensor cores: eight tcgen05.mma (K = 16
// each) from shared-memory operands, the fp32 accumulator in tensor memory.
// Both operands are K-major with the 128-byte swizzle: a tile of X arrives by
// two TMA boxes (coordinates 0-63 and 64-127, 128 rows of 128 bytes each), S
// is copied once per CTA into the same layout.  Roles (one persistent CTA
// per SM, 6 warps): warp 0 streams X tiles into a 4-stage ring, warp 1 owns
// the tensor memory and issues the MMAs (one thread), warps 2-5 are the
// epilogue: thread t of the four owns key row t of the tile (the tensor
// memory lane it may read), reads its m accumulators (tcgen05.ld), packs
// bit j = [dot_j >= 0] and takes the norm from the key's row in the staged
// tile.  The accumulator is double-buffered in tensor memory,
// so the MMAs of tile i + 1 run during the epilogue of tile i.  Every wait
// is bounded; on a timeout the CTA records VQ_DEVERR_WAIT_TIMEOUT, waits
// (bounded) for its copies in flight, frees its tensor memory and returns.
constexpr int QT_M = 128;                // keys per tile (MMA M)
constexpr int QT_STAGES = 4;             // X tiles in flight
constexpr int QT_HALF = QT_M * 128;      // one 64-coordinate half of a tile (bytes)
constexpr int QT_TILE = 2 * QT_HALF;     // 32 KB
constexpr int QT_EPI = 4;                // epilogue warps
constexpr int QT_THREADS = 32 * (2 + QT_EPI);

__host__ __device__ constexpr int qt_smem(int m)
{
    // 1024-byte alignment, the sketch (two halves of m rows x 128 bytes),
    // the ring, then the barriers and the tensor-memory address slot
    return 1024 + m * 256 + QT_STAGES * QT_TILE + 256;
}

// Bit j of the result: [v_j >= 0].  Adding +0 turns a negative zero into +0
// (round to nearest), so the complemented sign bit is exactly [v >= 0]; the
// funnel shift appends each sign below the ones already taken (j from 31
// down to 0 leaves bit j at position j).
__device__ __forceinline__ uint32_t qt_signs(const uint32_t (&r)[32])
{
    uint32_t w = 0u;
#pragma unroll
    for (int j = 31; j >= 0; --j) w = __funnelshift_l(__float_as_uint(__uint_as_float(r[j]) + 0.0f), w, 1);
    return ~w;
}

template <int W>
__global__ void __launch_bounds__(QT_THREADS, 1) qjl_encode_tc_kernel(const __grid_constant__ QjlEncodeParams p)
{
    constexpr int M = 32 * W;  // sketch rows (MMA N, accumulator columns per buffer)
    // tensor-memory columns: two accumulator buffers of M fp32 columns at a
    // power-of-two stride
    constexpr uint32_t ASTRIDE = M <= 32 ? 32 : M <= 64 ? 64 : M <= 128 ? 128 : 256;
    constexpr uint32_t TCOLS = 2 * ASTRIDE;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    unsigned char *base = smem_1k(smem_raw);
    unsigned char *ss = base;                        // sketch: half h at h * M * 128
    unsigned char *ring = base + M * 256;            // 1024-aligned (M is a multiple of 32)
    uint64_t *bars = reinterpret_cast<uint64_t *>(ring + QT_STAGES * QT_TILE);
    uint64_t *x_full = bars, *x_empty = bars + QT_STAGES;
    uint64_t *acc_full = bars + 2 * QT_STAGES, *acc_empty = acc_full + 2;
    volatile uint32_t *tslot = reinterpret_cast<volatile uint32_t *>(acc_empty + 2);
    volatile uint32_t *abort_flag = tslot + 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ntiles = (p.N + QT_M - 1) / QT_M;

    if (threadIdx.x == 0) {
        for (int s = 0; s < QT_STAGES; ++s) {
            mbar_init(&x_full[s], 1);
            mbar_init(&x_empty[s], QT_EPI);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&acc_full[a], 1);
            mbar_init(&acc_empty[a], QT_EPI);
        }
        *abort_flag = 0u;
        fence_mbar_init();
    }
    // the sketch into the swizzled K-major layout: 16-byte chunk c of row r
    {
        const uint4 *src = static_cast<const uint4 *>(p.s);
        for (int i = threadIdx.x; i < M * 16; i += blockDim.x) {
            const int r = i >> 4, c = i & 15;
            *reinterpret_cast<uint4 *>(ss + (c >> 3) * (M * 128) + swz128(r, c & 7)) = __ldg(src + i);
        }
        fence_proxy_async_smem();  // generic-proxy writes, read by the MMA (async proxy)
    }
    if (warp == 1) tmem_alloc(const_cast<uint32_t *>(tslot), TCOLS);
    qt_fence_before();
    __syncthreads();
    qt_fence_after();
    const uint32_t tmem = *tslot;

    if (warp == 0) {
        // ---- producer: X tiles into the ring
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            int i = 0;
            for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++i) {
                const int s = i % QT_STAGES;
                if (i >= QT_STAGES && !mbar_wait_bounded(&x_empty[s], (uint32_t)((i / QT_STAGES) - 1) & 1u)) {
                    atomicOr(&g_qjl_err, (unsigned)VQ_DEVERR_WAIT_TIMEOUT);
                    *abort_flag = 1u;
                    break;
                }
                if (*abort_flag) break;
                unsigned char *dst = ring + s * QT_TILE;
                mbar_arrive_expect_tx(&x_full[s], (uint32_t)QT_TILE);
                tma_load_2d(dst, &p.tmx, 0, t * QT_M, &x_full[s], pol);
                tma_load_2d(dst + QT_HALF, &p.tmx, 64, t * QT_M, &x_full[s], pol);
            }
            // the copies this CTA issued have all landed before it may exit
            for (int k = 0; k < QT_STAGES && k < i; ++k) {
                const int j = i - 1 - k;
                (void)mbar_wait_bounded(&x_full[j % QT_STAGES], (uint32_t)(j / QT_STAGES) & 1u);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---- MMA issue (one thread)
        if (lane == 0) {
            constexpr uint32_t IDESC = qt_idesc(M);
            const uint32_t sb = smem_u32(ss), rb = smem_u32(ring);
            int i = 0;
            for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++i) {
                const int s = i % QT_STAGES, a = i & 1;
                bool ok = mbar_wait_bounded(&x_full[s], (uint32_t)(i / QT_STAGES) & 1u);
                if (ok && i >= 2) ok = mbar_wait_bounded(&acc_empty[a], (uint32_t)((i >> 1) - 1) & 1u);
                if (!ok || *abort_flag) {
                    if (!ok) atomicOr(&g_qjl_err, (unsigned)VQ_DEVERR_WAIT_TIMEOUT);
                    *abort_flag = 1u;
                    break;
                }
                qt_fence_after();
                const uint32_t xa = rb + s * QT_TILE;
#pragma unroll
                for (int kb = 0; kb < 2; ++kb) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t ad = qt_desc(xa + kb * QT_HALF + kk * 32);
                        const uint64_t bd = qt_desc(sb + kb * (M * 128) + kk * 32);
                        qt_mma(tmem + (uint32_t)a * ASTRIDE, ad, bd, IDESC, (kb | kk) ? 1u : 0u);
                    }
                }
                qt_commit(&acc_full[a]);  // arrives when the MMAs are done (operands read, D written)
            }
        }
        __syncwarp();
    } else {
        // ---- epilogue: warp q = warp % 4 reads tensor-memory lanes 32 q .. 32 q + 31
        const int q = warp & 3;
        const int row = 32 * q + lane;
        int i = 0;
        for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++i) {
            const int s = i % QT_STAGES, a = i & 1;
            const bool ok = mbar_wait_bounded(&acc_full[a], (uint32_t)(i >> 1) & 1u);
            if (!__all_sync(FULL_MASK, ok) || *abort_flag) {
                if (!ok && lane == 0) atomicOr(&g_qjl_err, (unsigned)VQ_DEVERR_WAIT_TIMEOUT);
                *abort_flag = 1u;
                break;
            }
            qt_fence_after();
            uint32_t words[W];
#pragma unroll
            for (int w = 0; w < W; ++w) {
                uint32_t r[32];
                qt_ld32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)a * ASTRIDE + (uint32_t)(32 * w), r);
                qt_wait_ld();
                qt_hold(r);
                words[w] = qt_signs(r);
            }
            // the accumulator buffer is free for tile i + 2
            qt_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[a]);
            // the key's norm from its row of the staged tile (exact squares,
            // fp32 sums), then the stage is free
            const unsigned char *xt = ring + s * QT_TILE;
            float2 acc2 = make_float2(0.0f, 0.0f), acc3 = acc2;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 v = *reinterpret_cast<const uint4 *>(xt + h * QT_HALF + swz128(row, c));
                    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&u[j]));
                        if (j & 1) acc3 = __ffma2_rn(f, f, acc3);
                        else acc2 = __ffma2_rn(f, f, acc2);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&x_empty[s]);
            const int key = t * QT_M + row;
            if (key < p.N) {
                const float ss2 = (acc2.x + acc2.y) + (acc3.x + acc3.y);
                static_cast<__half *>(p.norms)[key] = __float2half_rn(__fsqrt_rn(ss2));
                uint32_t *dst = p.packed + (size_t)key * W;
                if constexpr (W % 4 == 0) {
#pragma unroll
                    for (int w = 0; w < W; w += 4)
                        *reinterpret_cast<uint4 *>(dst + w) = make_uint4(words[w], words[w + 1], words[w + 2], words[w + 3]);
                } else if constexpr (W % 2 == 0) {
#pragma unroll
                    for (int w = 0; w < W; w += 2) *reinterpret_cast<uint2 *>(dst + w) = make_uint2(words[w], words[w + 1]);
                } else {
#pragma unroll
                    for (int w = 0; w < W; ++w) dst[w] = words[w];
                }
            }
        }
    }

    // every tcgen05.ld has completed (wait::ld) and every MMA has been
    // consumed or abandoned: free the tensor memory
    qt_fence_before();
    __syncthreads();
    qt_fence_after();
    if (warp == 1) tmem_free(tmem, TCOLS);
}

}  // namespace

cudaError_t launch_qjl_encode(const QjlEncodeParams &p0, cudaStream_t stream)
{
    if (p0.N <= 0) return cudaSuccess;
    QjlEncodeParams p = p0;
    {
        const uint64_t dims[2] = {(uint64_t)D, (uint64_t)p.N};
        const uint64_t strides[1] = {(uint64_t)D * 2};
        const uint32_t box[2] = {64u, (uint32_t)QT_M};
        if (!encode_tmap_f16(&p.tmx, p.x, 2, dims, strides, box, true, true)) return cudaErrorInvalidValue;
    }
    const int smem = qt_smem(p.m);
    void (*kern)(QjlEncodeParams) = nullptr;
    switch (p.m / 32) {
    case 1: kern = qjl_encode_tc_kernel<1>; break;
    case 2: kern = qjl_encode_tc_kernel<2>; break;
    case 3: kern = qjl_encode_tc_kernel<3>; break;
    case 4: kern = qjl_encode_tc_kernel<4>; break;
    case 5: kern = qjl_encode_tc_kernel<5>; break;
    case 6: kern = qjl_encode_tc_kernel<6>; break;
    case 7: kern = qjl_encode_tc_kernel<7>; break;
    case 8: kern = qjl_encode_tc_kernel<8>; break;
    default: return cudaErrorInvalidValue;
    }
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    // one CTA per SM (it holds up to 512 tensor-memory columns)
    const int ntiles = (p.N + QT_M - 1) / QT_M;
    const int grid = ntiles < sm_count() ? ntiles : sm_count();
    kern<<<grid, QT_THREADS, smem, stream>>>(p);
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
