// kivi.cu - KIVI asymmetric min/max group quantize+pack and unpack+dequant
// kernels for sm_103a.
//
// The quantizers' device code (method, exactness and layout notes) is in
// kivi_quant.cuh; here are their kernels, the dequant kernels and the
// launchers.  Dequant: one fp16x2 fused multiply-add per element pair,
// q * scale + zero rounded once from its exact value (fma.rn.f16x2), the code
// entering exactly as (1024 + q) - 1024 in fp16.
#include <cuda_fp16.h>

#include "device_common.cuh"
#include "launch.h"

namespace vq {
VQ_DEFINE_ERROR_WORD(g_kivi_err);
}  // namespace vq

#define VQ_KIVI_ERR g_kivi_err
#include "kivi_quant.cuh"

namespace vq {

namespace {

template <int BITS, int G>
__global__ void __launch_bounds__(VAL_WARPS * 32, 1) kivi_values_kernel(const __grid_constant__ KiviQuantParams p)
{
    kivi_values_body<BITS, G, VAL_WARPS>(p, blockIdx.x, gridDim.x);
}

template <int BITS, int G>
__global__ void __launch_bounds__(key_warps<BITS, G>() * 32, 1) kivi_keys_kernel(const __grid_constant__ KiviQuantParams p)
{
    kivi_keys_body<BITS, G, key_warps<BITS, G>()>(p, blockIdx.x, gridDim.x);
}

// ------------------------------------------------------------ dequant

constexpr int DQ_THREADS = 256;

// Values: two threads per row: lane l works on row l & 15 of a 16-row block
// and on channels [64h, 64h + 64), h = l >> 4.  The words of a block
// (contiguous in memory) arrive by one bulk copy into a per-warp 3-stage
// ring; scale/zero of the lane's groups are read one block ahead.  Each
// element is one fp16x2 fused multiply-add, q s + z rounded once from its
// exact value (the definition of the dequant), two elements per instruction:
// codes k and k + E/2 of a word sit at bits b k and b k + 16, so one shift and
// one mask-or put both into the mantissas of 1024 + q, a subtract of 1024
// leaves q exactly, and byte permutes pair the results as consecutive
// elements.  The fp16 half rows are staged in shared memory and written out
// coalesced (the 16 rows of a block are contiguous).
constexpr int VDQ_WARPS = 24;
constexpr int VDQ_STAGES = 3;
constexpr int VDR = 16;  // rows per block
__host__ __device__ constexpr int vdq_stage(int bits) { return VDR * (D * bits / 32) * 4; }
__host__ __device__ constexpr int vdq_warp_bytes(int bits) { return VDQ_STAGES * vdq_stage(bits) + VDR * ROW_STRIDE; }
__host__ __device__ constexpr int vdq_smem(int bits) { return VDQ_WARPS * (vdq_warp_bytes(bits) + VDQ_STAGES * 8); }

template <int BITS, int G>
__global__ void __launch_bounds__(VDQ_WARPS * 32, 1) kivi_values_dequant_kernel(const __grid_constant__ KiviDequantParams p)
{
    constexpr int E = 32 / BITS;
    constexpr int W = D * BITS / 32;
    constexpr int WL = W / 2;              // words of a half row
    constexpr int NGD = D / G;
    constexpr int GL = G < 64 ? G : 64;    // group members held by one thread
    constexpr int NGL = 64 / GL;           // groups (or group halves) per thread
    constexpr uint32_t MASK = (1u << BITS) - 1u;
    static_assert(GL % E == 0, "a packed word lies inside one group");
    constexpr int STG = vdq_stage(BITS);
    constexpr int WB = vdq_warp_bytes(BITS);
    extern __shared__ __align__(128) unsigned char smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int rr = lane & 15, hh = lane >> 4;
    unsigned char *wbuf = smem + warp * WB;
    unsigned char *obuf = wbuf + VDQ_STAGES * STG;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + VDQ_WARPS * WB) + warp * VDQ_STAGES;
    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < VDQ_STAGES; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    __syncwarp();
    const uint64_t pol = l2_policy_evict_first();
    const int N = p.BH * p.S_q;
    const int nblk = (N + VDR - 1) / VDR;
    const int gw = blockIdx.x * VDQ_WARPS + warp;
    const int tw = gridDim.x * VDQ_WARPS;
    auto issue = [&](int blk, int s) {
        if (lane == 0) {
            const int r0 = blk * VDR;
            const uint32_t bytes = (uint32_t)(min(VDR, N - r0) * W * 4);
            mbar_arrive_expect_tx(&bars[s], bytes);
            bulk_g2s(wbuf + s * STG, p.packed + (size_t)r0 * W, bytes, &bars[s], pol);
        }
    };
#pragma unroll
    for (int s = 0; s < VDQ_STAGES; ++s) {
        const int blk = gw + s * tw;
        if (blk < nblk) issue(blk, s);
    }
    const __half *scp = static_cast<const __half *>(p.scale);
    const __half *zrp = static_cast<const __half *>(p.zero);
    // scale/zero of this lane's groups, loaded one block ahead
    const int j0 = G == 128 ? 0 : hh * NGL;
    __half sh[NGL], zh[NGL];
    auto load_sz = [&](int blk) {
        const int row = blk * VDR + rr;
        const bool ok = blk < nblk && row < N;
#pragma unroll
        for (int j = 0; j < NGL; ++j) {
            sh[j] = ok ? scp[(size_t)row * NGD + j0 + j] : __float2half_rn(0.0f);
            zh[j] = ok ? zrp[(size_t)row * NGD + j0 + j] : __float2half_rn(0.0f);
        }
    };
    load_sz(gw);
    for (int it = 0;; ++it) {
        const int blk = gw + it * tw;
        if (blk >= nblk) break;
        const int s = it % VDQ_STAGES;
        __half2 s2[NGL], z2[NGL];
#pragma unroll
        for (int j = 0; j < NGL; ++j) {
            s2[j] = __half2half2(sh[j]);
            z2[j] = __half2half2(zh[j]);
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
        const uint32_t *wrow = reinterpret_cast<const uint32_t *>(wbuf + s * STG) + rr * W + hh * WL;
        uint32_t wd[WL];
        if constexpr (WL == 2) {
            const uint2 a = *reinterpret_cast<const uint2 *>(wrow);
            wd[0] = a.x; wd[1] = a.y;
        } else {
#pragma unroll
            for (int i = 0; i < WL; i += 4) {
                const uint4 a = *reinterpret_cast<const uint4 *>(wrow + i);
                wd[i] = a.x; wd[i + 1] = a.y; wd[i + 2] = a.z; wd[i + 3] = a.w;
            }
        }
        uint4 *orow = reinterpret_cast<uint4 *>(obuf + rr * ROW_STRIDE + hh * 128);
        const __half2 k1024 = __float2half2_rn(1024.0f);
#pragma unroll
        for (int i = 0; i < WL; ++i) {
            const int jl = (i * E) / GL;  // a word lies inside one group (GL >= E)
            uint32_t r[E / 2];
#pragma unroll
            for (int k = 0; k < E / 2; ++k) {
                const uint32_t x = ((wd[i] >> (BITS * k)) & (MASK | (MASK << 16))) | 0x64006400u;
                const __half2 q2 = __hsub2(*reinterpret_cast<const __half2 *>(&x), k1024);
                const __half2 v2 = __hfma2(q2, s2[jl], z2[jl]);
                r[k] = *reinterpret_cast<const uint32_t *>(&v2);
            }
            // r[k] = (element k, element k + E/2) of the word -> consecutive pairs
            uint32_t o[E / 2];
#pragma unroll
            for (int j = 0; j < E / 4; ++j) {
                o[j] = __byte_perm(r[2 * j], r[2 * j + 1], 0x5410);
                o[E / 4 + j] = __byte_perm(r[2 * j], r[2 * j + 1], 0x7632);
            }
#pragma unroll
            for (int c = 0; c < E / 8; ++c)
                orow[(i * E) / 8 + c] = make_uint4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
        }
        __syncwarp();
        fence_proxy_async_smem();
        {
            const int nb = blk + VDQ_STAGES * tw;
            if (nb < nblk) issue(nb, s);
        }
        const int nrows = min(VDR, N - blk * VDR);
        uint4 *gout = reinterpret_cast<uint4 *>(static_cast<__half *>(p.out) + (size_t)blk * VDR * D);
#pragma unroll
        for (int i = 0; i < VDR / 2; ++i) {
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
        // scale / zero of channels (4l, 4l + 1) and (4l + 2, 4l + 3) as fp16 pairs
        const __half2 sa = *reinterpret_cast<const __half2 *>(&sraw.x), sb = *reinterpret_cast<const __half2 *>(&sraw.y);
        const __half2 za = *reinterpret_cast<const __half2 *>(&zraw.x), zb = *reinterpret_cast<const __half2 *>(&zraw.y);
        const __half2 k1024 = __float2half2_rn(1024.0f);
        // up to four word rows of the tile in flight before any is used (a
        // ragged last group's pad words exist and hold code 0)
        constexpr int KB = WG < 4 ? WG : 4;
        for (int k0 = 0; k0 < WG; k0 += KB) {
            uint4 wvs[KB];
#pragma unroll
            for (int kk = 0; kk < KB; ++kk)
                wvs[kk] = __ldg(reinterpret_cast<const uint4 *>(p.packed + ((size_t)tile * WG + k0 + kk) * D + 4 * lane));
#pragma unroll
            for (int kk = 0; kk < KB; ++kk) {
                const int k = k0 + kk;
                const uint4 wv = wvs[kk];
                // the two channels of a pair side by side: tokens j < E/2 from the
                // low halves of their words, the others from the high halves
                const uint32_t alo = __byte_perm(wv.x, wv.y, 0x5410), ahi = __byte_perm(wv.x, wv.y, 0x7632);
                const uint32_t blo = __byte_perm(wv.z, wv.w, 0x5410), bhi = __byte_perm(wv.z, wv.w, 0x7632);
#pragma unroll 4
                for (int j = 0; j < E; ++j) {
                    const int i = k * E + j;
                    if (i >= ntok) break;
                    // q s + z rounded once from its exact value: one fp16x2 FMA
                    // per channel pair (codes as the mantissas of 1024 + q)
                    const int sh = BITS * (j % (E / 2));
                    const uint32_t xa = (((j < E / 2 ? alo : ahi) >> sh) & (MASK | (MASK << 16))) | 0x64006400u;
                    const uint32_t xb = (((j < E / 2 ? blo : bhi) >> sh) & (MASK | (MASK << 16))) | 0x64006400u;
                    const __half2 ha = __hfma2(__hsub2(*reinterpret_cast<const __half2 *>(&xa), k1024), sa, za);
                    const __half2 hb = __hfma2(__hsub2(*reinterpret_cast<const __half2 *>(&xb), k1024), sb, zb);
                    *reinterpret_cast<uint2 *>(static_cast<__half *>(p.out) + ((size_t)bh * p.S_q + g * G + i) * D + 4 * lane) =
                        make_uint2(*reinterpret_cast<const uint32_t *>(&ha), *reinterpret_cast<const uint32_t *>(&hb));
                }
            }
        }
    }
}

// ------------------------------------------------------------ launchers

template <int BITS, int G>
cudaError_t launch_q(const KiviQuantParams &p0, bool per_channel, cudaStream_t stream)
{
    const int sms = sm_count();
    KiviQuantParams p = p0;
    if (!prepare_kivi_quant(p, per_channel)) return cudaErrorInvalidValue;
    if (per_channel) {
        auto kern = kivi_keys_kernel<BITS, G>;
        constexpr int smem = key_smem<BITS, G>();
        constexpr int warps = key_warps<BITS, G>();
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        const int ntiles = p.B * p.H * ((p.S_q + G - 1) / G) * 2;
        int grid = (ntiles + warps - 1) / warps;
        if (grid > sms) grid = sms;
        if (grid < 1) grid = 1;
        kern<<<grid, warps * 32, smem, stream>>>(p);
    } else {
        auto kern = kivi_values_kernel<BITS, G>;
        constexpr int smem = val_smem();
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        const int nblk = p.B * p.H * ((p.S_q + VROWS - 1) / VROWS);
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
    if (per_channel) {
        // one resident wave: as many CTAs as fit on the SMs at once (the warps
        // stride over the tiles), so that no partial second wave forms the tail
        static int per_sm = 0;
        if (per_sm == 0) {
            int b = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kivi_keys_dequant_kernel<BITS, G>, DQ_THREADS, 0) !=
                    cudaSuccess ||
                b < 1)
                b = 1;
            per_sm = b;
        }
        const int cap = sm_count() * per_sm;
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
        const int nblk = (p.BH * p.S_q + VDR - 1) / VDR;
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

bool prepare_kivi_quant(KiviQuantParams &p, bool per_channel)
{
    const int G = p.group;
    p.divH = make_fastdiv((uint32_t)p.H);
    p.divBlk = make_fastdiv((uint32_t)(per_channel ? (p.S_q + G - 1) / G : (p.S_q + VROWS - 1) / VROWS));
    const uint64_t dims[3] = {(uint64_t)D, (uint64_t)p.S, (uint64_t)p.B * p.H};
    const uint64_t strides[2] = {(uint64_t)D * 2, (uint64_t)p.S * D * 2};
    const uint32_t box[3] = {64u, per_channel ? (uint32_t)G : (uint32_t)VROWS, 1u};
    // keys: a warp loads one 128-byte half of each token row (the other
    // half belongs to another warp's tile): no 256-byte promotion
    return encode_tmap_f16(&p.tmap, p.x, 3, dims, strides, box, !per_channel, !per_channel);
}

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
