// rvq_generic.cu - TurboQuantRVQ encode+pack and unpack+dequant at every head
// width and bit count the pages test (VeloxQuant-MLX blog, tag "rvq",
// "Bit-exactness, checked the boring way": D in {8, ..., 256}, b in
// {1, 2, 3, 4}), for the shapes the D = 128, b in {1, 2, 4} kernels of rvq.cu
// do not serve.  Same method as rvq.cu ("The pipeline, as it actually runs"):
// n = ||x||, y = H (x / n) / sqrt(D), i1 = #{y > b1_k}, r = y - c1[i1],
// i2 = #{r > b2_k}, both streams packed LSB first with E = floor(32/b) codes
// per word (b = 3: 10 codes, the top two bits zero).
//
// Layout: one warp step holds RPW = 32 / LPR rows, LPR = min(D, 32) lanes per
// row, C = D / LPR consecutive coordinates per lane (coordinate ll * C + j).
// The Walsh-Hadamard butterflies run over j in registers and over the lane
// bits by shuffles.  Codes go through a per-warp byte buffer in shared memory
// so that lanes can assemble words whose codes straddle lanes (b = 3).
// Exactness: the row is computed in fp32 (the norm from a double-float sum of
// the exact squares, no binary64 on the common path: that pipe is slow on
// this GPU); a step with any value within the guard band of a boundary (or a
// zero row) is recomputed by the same code in binary64 (the fp16 inputs are
// exact there; the rounding then differs from the oracle's only far inside
// its tie band).
#include <cuda_fp16.h>

#include "device_common.cuh"
#include "launch.h"

namespace vq {

namespace {

VQ_DEFINE_ERROR_WORD(g_gen_err);

constexpr int GEN_WARPS = 8;

template <int D>
struct GenShape {
    static constexpr int LPR = D < 32 ? D : 32;  // lanes per row
    static constexpr int C = D / LPR;            // coordinates per lane
    static constexpr int RPW = 32 / LPR;         // rows per warp step
};

// Walsh-Hadamard transform (Sylvester order, unnormalised) of a row spread
// over LPR lanes: lower = a + b, upper = a - b at every stage.
template <typename T, int C, int LPR>
__device__ __forceinline__ void gen_wht(T (&a)[C], int ll)
{
#pragma unroll
    for (int h = 1; h < C; h <<= 1)
#pragma unroll
        for (int j = 0; j < C; ++j)
            if ((j & h) == 0) {
                const T u = a[j], v = a[j + h];
                a[j] = u + v;
                a[j + h] = u - v;
            }
#pragma unroll
    for (int m = 1; m < LPR; m <<= 1) {
        const bool upper = (ll & m) != 0;
#pragma unroll
        for (int j = 0; j < C; ++j) {
            const T o = __shfl_xor_sync(FULL_MASK, a[j], m);
            a[j] = upper ? (o - a[j]) : (a[j] + o);
        }
    }
}

// Both stage codes of this lane's C values and the smallest distance to a
// boundary (stage 1 on y, stage 2 on the residual).  The centroid c1[i1] is
// read by shuffle from tcen = c1[lane mod 2^b].
template <typename T, int BITS, int C>
__device__ __forceinline__ void gen_quant(const RvqGenericParams &p, const T (&y)[C], float tcen,
                                          uint32_t (&q1)[C], uint32_t (&q2)[C], T &m)
{
    constexpr int L = 1 << BITS;
#pragma unroll
    for (int j = 0; j < C; ++j) {
        int i1 = 0;
#pragma unroll
        for (int k = 0; k < L - 1; ++k) {
            const T b = (T)p.b1[k];
            i1 += y[j] > b ? 1 : 0;
            const T d = y[j] - b;
            m = fmin(m, d < (T)0 ? -d : d);
        }
        const T r = y[j] - (T)__shfl_sync(FULL_MASK, tcen, i1);
        int i2 = 0;
#pragma unroll
        for (int k = 0; k < L - 1; ++k) {
            const T b = (T)p.b2[k];
            i2 += r > b ? 1 : 0;
            const T d = r - b;
            m = fmin(m, d < (T)0 ? -d : d);
        }
        q1[j] = (uint32_t)i1;
        q2[j] = (uint32_t)i2;
    }
}

// Destination row of source row `row`; false if its batch offset is invalid.
__device__ __forceinline__ bool gen_dst_row(const RvqGenericParams &p, int row, size_t &drow)
{
    const int bh = row / p.S;
    const int s = row - bh * p.S;
    int off = 0;
    if (p.dst_off != nullptr) {
        off = __ldg(p.dst_off + bh / p.H);
        if (off < 0 || off > p.S_dst - p.S) {
            atomicOr(&g_gen_err, (unsigned)VQ_DEVERR_BAD_OFFSET);
            return false;
        }
    }
    drow = (size_t)bh * p.S_dst + off + s;
    return true;
}

template <int C>
__device__ __forceinline__ void load_halves(const __half *src, float (&x)[C])
{
    if constexpr (C == 1) {
        x[0] = __half2float(*src);
    } else if constexpr (C == 2) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(src));
        x[0] = f.x;
        x[1] = f.y;
    } else {
#pragma unroll
        for (int j = 0; j < C; j += 4) {
            const uint2 u = *reinterpret_cast<const uint2 *>(src + j);
            const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&u.x));
            const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&u.y));
            x[j] = a.x;
            x[j + 1] = a.y;
            x[j + 2] = b.x;
            x[j + 3] = b.y;
        }
    }
}

// sqrt(D) as the nearest fp32 (D a power of two from 8 to 256)
template <int D>
__host__ __device__ constexpr float sqrt_d_f()
{
    return D == 8 ? 2.8284271247461903f : D == 16 ? 4.0f : D == 32 ? 5.656854249492381f : D == 64 ? 8.0f
         : D == 128 ? 11.313708498984761f : 16.0f;
}

template <int D, int BITS>
__global__ void __launch_bounds__(GEN_WARPS * 32) rvq_generic_encode_kernel(const __grid_constant__ RvqGenericParams p)
{
    using S = GenShape<D>;
    constexpr int LPR = S::LPR, C = S::C, RPW = S::RPW;
    constexpr int L = 1 << BITS;
    constexpr int E = 32 / BITS;
    constexpr int W = (D + E - 1) / E;
    __shared__ uint8_t cbuf[GEN_WARPS][2][32 * C];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rl = lane / LPR, ll = lane % LPR;
    const float tcen = p.c1[lane & (L - 1)];
    const double inv_sqrt_d = 1.0 / sqrt((double)D);
    const int nsteps = (p.N + RPW - 1) / RPW;
    for (int step = blockIdx.x * GEN_WARPS + warp; step < nsteps; step += gridDim.x * GEN_WARPS) {
        const int row = step * RPW + rl;
        const bool valid = row < p.N;
        float x[C];
        if (valid) {
            load_halves<C>(static_cast<const __half *>(p.x) + (size_t)row * D + ll * C, x);
        } else {
#pragma unroll
            for (int j = 0; j < C; ++j) x[j] = 0.0f;
        }
        // row norm: squares of fp16 values are exact in fp32, summed as a
        // double-float (two_sum), the square root corrected once: the norm is
        // the correctly rounded fp32 of the exact one but for rare ties, with
        // no binary64 arithmetic (a slow pipe on this GPU) on the common path
        float qh = 0.0f, ql = 0.0f;
#pragma unroll
        for (int j = 0; j < C; ++j) {
            float t, e;
            two_sum(qh, x[j] * x[j], t, e);
            qh = t;
            ql += e;
        }
#pragma unroll
        for (int m = 1; m < LPR; m <<= 1) {
            const float oh = __shfl_xor_sync(FULL_MASK, qh, m);
            const float ol = __shfl_xor_sync(FULL_MASK, ql, m);
            float t, e;
            two_sum(qh, oh, t, e);
            e += ql + ol;
            fast_two_sum(t, e, qh, ql);
        }
        float nh = 0.0f, nl = 0.0f;
        if (qh > 0.0f) {
            nh = __fsqrt_rn(qh);
            nl = __fdiv_rn(fmaf(-nh, nh, qh) + ql, 2.0f * nh);
        }
        const float nrm = __fadd_rn(nh, nl);

        // fp32 fast path
        uint32_t q1[C], q2[C];
        {
            float y[C];
#pragma unroll
            for (int j = 0; j < C; ++j) y[j] = x[j];
            gen_wht<float, C, LPR>(y, ll);
            const float inv = qh > 0.0f ? __frcp_rn(nrm * (float)sqrt_d_f<D>()) : 0.0f;
#pragma unroll
            for (int j = 0; j < C; ++j) y[j] *= inv;
            float m = __int_as_float(0x7f800000);
            gen_quant<float, BITS, C>(p, y, tcen, q1, q2, m);
            const bool flag = valid && (!(m >= p.guard) || !(qh > 0.0f));
            if (__any_sync(FULL_MASK, flag)) {
                // binary64 recompute of the whole step (uniform across the warp)
                const double n64 = (double)nh + (double)nl;
                double u[C];
#pragma unroll
                for (int j = 0; j < C; ++j) u[j] = n64 > 0.0 ? (double)x[j] / n64 : 0.0;
                gen_wht<double, C, LPR>(u, ll);
#pragma unroll
                for (int j = 0; j < C; ++j) u[j] *= inv_sqrt_d;
                double md = __longlong_as_double(0x7ff0000000000000ll);
                gen_quant<double, BITS, C>(p, u, tcen, q1, q2, md);
            }
        }

        // pack: codes through shared memory, then lane i < RPW * W assembles
        // word i % W of row i / W of this step, for each stream
#pragma unroll
        for (int j = 0; j < C; ++j) {
            cbuf[warp][0][lane * C + j] = (uint8_t)q1[j];
            cbuf[warp][1][lane * C + j] = (uint8_t)q2[j];
        }
        __syncwarp();
        if (lane < RPW * W) {
            const int r = lane / W, w = lane - r * W;
            const int orow = step * RPW + r;
            size_t drow = 0;
            if (orow < p.N && gen_dst_row(p, orow, drow)) {
                uint32_t a = 0u, b = 0u;
#pragma unroll
                for (int j = 0; j < E; ++j) {
                    const int i = w * E + j;
                    if (i < D) {
                        a |= (uint32_t)cbuf[warp][0][r * D + i] << (j * BITS);
                        b |= (uint32_t)cbuf[warp][1][r * D + i] << (j * BITS);
                    }
                }
                p.p1[drow * W + w] = a;
                p.p2[drow * W + w] = b;
            }
        }
        if (valid && ll == 0) {
            size_t drow = 0;
            if (gen_dst_row(p, row, drow)) p.norms[drow] = nrm;
        }
        __syncwarp();
    }
}

template <int D, int BITS>
__global__ void __launch_bounds__(GEN_WARPS * 32) rvq_generic_decode_kernel(const __grid_constant__ RvqGenericParams p)
{
    using S = GenShape<D>;
    constexpr int LPR = S::LPR, C = S::C, RPW = S::RPW;
    constexpr int L = 1 << BITS;
    constexpr int E = 32 / BITS;
    constexpr int W = (D + E - 1) / E;
    __shared__ uint32_t wbuf[GEN_WARPS][2][32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rl = lane / LPR, ll = lane % LPR;
    const float tc1 = p.c1[lane & (L - 1)];
    const float tc2 = p.c2[lane & (L - 1)];
    const float rsd = (float)(1.0 / sqrt((double)D));
    const int nsteps = (p.N + RPW - 1) / RPW;
    for (int step = blockIdx.x * GEN_WARPS + warp; step < nsteps; step += gridDim.x * GEN_WARPS) {
        // the step's words (RPW rows x W words of each stream; rows are contiguous)
        const int nrows = min(RPW, p.N - step * RPW);
        if (lane < nrows * W) {
            wbuf[warp][0][lane] = __ldg(p.p1 + (size_t)step * RPW * W + lane);
            wbuf[warp][1][lane] = __ldg(p.p2 + (size_t)step * RPW * W + lane);
        }
        __syncwarp();
        const int row = step * RPW + rl;
        const bool valid = row < p.N;
        float v[C];
#pragma unroll
        for (int j = 0; j < C; ++j) {
            const int i = ll * C + j;
            const int w = i / E, sh = (i - w * E) * BITS;
            const uint32_t a = valid ? wbuf[warp][0][rl * W + w] : 0u;
            const uint32_t b = valid ? wbuf[warp][1][rl * W + w] : 0u;
            v[j] = __shfl_sync(FULL_MASK, tc1, (int)((a >> sh) & (L - 1))) +
                   __shfl_sync(FULL_MASK, tc2, (int)((b >> sh) & (L - 1)));
        }
        gen_wht<float, C, LPR>(v, ll);
        const float n = valid ? __ldg(p.norms + row) : 0.0f;
        const float sc = n * rsd;
        if (valid) {
            __half *dst = static_cast<__half *>(p.out) + (size_t)row * D + ll * C;
            if constexpr (C == 1) {
                dst[0] = __float2half_rn(v[0] * sc);
            } else {
#pragma unroll
                for (int j = 0; j < C; j += 2)
                    *reinterpret_cast<__half2 *>(dst + j) = __floats2half2_rn(v[j] * sc, v[j + 1] * sc);
            }
        }
        __syncwarp();
    }
}

template <int D, int BITS>
cudaError_t launch_gen(const RvqGenericParams &p, bool encode, cudaStream_t stream)
{
    constexpr int RPW = GenShape<D>::RPW;
    const int nsteps = (p.N + RPW - 1) / RPW;
    int grid = (nsteps + GEN_WARPS - 1) / GEN_WARPS;
    const int cap = sm_count() * 8;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    if (encode)
        rvq_generic_encode_kernel<D, BITS><<<grid, GEN_WARPS * 32, 0, stream>>>(p);
    else
        rvq_generic_decode_kernel<D, BITS><<<grid, GEN_WARPS * 32, 0, stream>>>(p);
    return cudaGetLastError();
}

template <int D>
cudaError_t dispatch_gen_bits(const RvqGenericParams &p, int bits, bool encode, cudaStream_t stream)
{
    switch (bits) {
    case 1: return launch_gen<D, 1>(p, encode, stream);
    case 2: return launch_gen<D, 2>(p, encode, stream);
    case 3: return launch_gen<D, 3>(p, encode, stream);
    case 4: return launch_gen<D, 4>(p, encode, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_rvq_generic(const RvqGenericParams &p, int bits, bool encode, cudaStream_t stream)
{
    if (p.N <= 0) return cudaSuccess;
    switch (p.D) {
    case 8: return dispatch_gen_bits<8>(p, bits, encode, stream);
    case 16: return dispatch_gen_bits<16>(p, bits, encode, stream);
    case 32: return dispatch_gen_bits<32>(p, bits, encode, stream);
    case 64: return dispatch_gen_bits<64>(p, bits, encode, stream);
    case 128: return dispatch_gen_bits<128>(p, bits, encode, stream);
    case 256: return dispatch_gen_bits<256>(p, bits, encode, stream);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t gen_take_device_error(unsigned *bits, cudaStream_t stream)
{
    *bits = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(bits, g_gen_err, sizeof(unsigned), 0, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    if (*bits) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbolAsync(g_gen_err, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice, stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    }
    return e;
}

}  // namespace vq
