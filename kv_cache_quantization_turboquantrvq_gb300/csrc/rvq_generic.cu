// rvq_generic.cu - TurboQuantRVQ encode+pack and unpack+dequant at every head
// width and bit count the pages test (VeloxQuant-MLX blog, tag "rvq",
// "Bit-exactness, checked the boring way": D in {8, ..., 256}, b in
// {1, 2, 3, 4}), for the shapes the D = 128, b in {1, 2, 4} kernels of rvq.cu
// do not serve.  Same method as rvq.cu ("The pipeline, as it actually runs"):
// n = ||x||, y = H (x / n) / sqrt(D), i1 = #{y > b1_k}, r = y - c1[i1],
// i2 = #{r > b2_k}, both streams packed LSB first with E = floor(32/b) codes
// per word (b = 3: 10 codes, the top two bits zero).
//
// Layout: one warp step holds RPW = 32 / LPR rows; a lane holds C = 8
// consecutive coordinates of one row (one 16-byte load), LPR = D / 8 lanes per
// row.  The Walsh-Hadamard butterflies run over the three coordinate bits in
// registers and over the lane bits by shuffles.  The quantizer counts
// boundaries by a binary search over the (validated ascending) boundaries in
// shared memory, and its margin is the distance to the two neighbouring
// boundaries.  Codes go through a per-warp byte buffer in shared memory so
// that lanes can assemble words whose codes straddle lanes (b = 3).
// Exactness: the fast path runs in fp32 (the norm from a double-float sum of
// the exact squares); its error on y is at most (log2 D + 2.5) fp32 units,
// below the 1e-6 guard band.  A step with any value inside the band (or a zero
// row) is recomputed exactly: the row split into three pieces on power-of-two
// grids whose transforms are exact in fp32, S = H x summed as a double-float,
// y = S / (n sqrt(D)) and the residual as double-floats (about 2^-46
// relative), the decisions taken on those.  No binary64 arithmetic (a slow
// pipe on this GPU) anywhere.
#include <cuda_fp16.h>

#include "device_common.cuh"
#include "launch.h"

namespace vq {

namespace {

VQ_DEFINE_ERROR_WORD(g_gen_err);

constexpr int GEN_WARPS = 8;

template <int D>
struct GenShape {
    static constexpr int C = 8;           // consecutive coordinates per lane
    static constexpr int LPR = D / C;     // lanes per row (1 .. 32)
    static constexpr int RPW = 32 / LPR;  // rows per warp step
};

// Walsh-Hadamard transform (Sylvester order, unnormalised) of a row spread
// over LPR lanes: lower = a + b, upper = a - b at every stage.
template <int C, int LPR>
__device__ __forceinline__ void gen_wht(float (&a)[C], int ll)
{
#pragma unroll
    for (int h = 1; h < C; h <<= 1)
#pragma unroll
        for (int j = 0; j < C; ++j)
            if ((j & h) == 0) {
                const float u = a[j], v = a[j + h];
                a[j] = __fadd_rn(u, v);
                a[j + h] = __fsub_rn(u, v);
            }
#pragma unroll
    for (int m = 1; m < LPR; m <<= 1) {
        const bool upper = (ll & m) != 0;
#pragma unroll
        for (int j = 0; j < C; ++j) {
            const float o = __shfl_xor_sync(FULL_MASK, a[j], m);
            a[j] = upper ? __fsub_rn(o, a[j]) : __fadd_rn(a[j], o);
        }
    }
}

// Books in shared memory: sb[0] = -inf, sb[1 .. L-1] = the boundaries
// (ascending), sb[L] = +inf; centroids c1.
struct GenBooks {
    float b1[17], b2[17], c1[16];
};

// #{k : v > b_k} by binary search; sb as above.
template <int BITS>
__device__ __forceinline__ int gen_count(const float *sb, float v)
{
    int i = 0;
#pragma unroll
    for (int s = (1 << BITS) >> 1; s >= 1; s >>= 1)
        if (v > sb[i + s]) i += s;
    return i;
}

// Both codes of one value on the fp32 fast path, and the distance to the
// nearest boundary of either stage folded into m.
template <int BITS>
__device__ __forceinline__ void gen_quant_fast(const GenBooks &bk, float y, uint32_t &q1, uint32_t &q2, float &m)
{
    const int i1 = gen_count<BITS>(bk.b1, y);
    m = fminf(m, fminf(__fsub_rn(y, bk.b1[i1]), __fsub_rn(bk.b1[i1 + 1], y)));
    const float r = __fsub_rn(y, bk.c1[i1]);
    const int i2 = gen_count<BITS>(bk.b2, r);
    m = fminf(m, fminf(__fsub_rn(r, bk.b2[i2]), __fsub_rn(bk.b2[i2 + 1], r)));
    q1 = (uint32_t)i1;
    q2 = (uint32_t)i2;
}

// [vh + vl > b] for a double-float v: vh - b is exact when the two are close
// (Sterbenz) and far larger than vl otherwise.
__device__ __forceinline__ bool df_above(float vh, float vl, float b)
{
    return __fadd_rn(__fsub_rn(vh, b), vl) > 0.0f;
}

template <int BITS>
__device__ __forceinline__ int gen_count_df(const float *sb, float vh, float vl)
{
    int i = 0;
#pragma unroll
    for (int s = (1 << BITS) >> 1; s >= 1; s >>= 1)
        if (df_above(vh, vl, sb[i + s])) i += s;
    return i;
}

// sqrt(D) as a double-float (D a power of two from 8 to 256): 2^(k/2), times
// sqrt(2) for odd k
template <int D>
__host__ __device__ constexpr int log2_d()
{
    return D == 8 ? 3 : D == 16 ? 4 : D == 32 ? 5 : D == 64 ? 6 : D == 128 ? 7 : 8;
}
constexpr float SQRT2_HI = 1.41421353816986083984375f;  // fp32 nearest to sqrt(2)
constexpr float SQRT2_LO = 2.4203234971764687e-08f;  // sqrt(2) - SQRT2_HI, rounded

// sqrt(D) as the nearest fp32
template <int D>
__host__ __device__ constexpr float sqrt_d_f()
{
    return (log2_d<D>() & 1) ? SQRT2_HI * (float)(1 << (log2_d<D>() >> 1)) : (float)(1 << (log2_d<D>() >> 1));
}

// Exact recompute of this lane's C codes (see the header): x the lane's fp16
// values as fp32, (nh, nl) the row norm as a double-float.
template <int D, int BITS>
__device__ __forceinline__ void gen_exact(const GenBooks &bk, const float (&x)[8], float nh, float nl, int ll,
                                         uint32_t (&q1)[8], uint32_t (&q2)[8])
{
    using S = GenShape<D>;
    constexpr int C = S::C, LPR = S::LPR;
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < C; ++j) amax = fmaxf(amax, fabsf(x[j]));
#pragma unroll
    for (int m = 1; m < LPR; m <<= 1) amax = fmaxf(amax, __shfl_xor_sync(FULL_MASK, amax, m));
    // (the whole warp runs this: the transforms shuffle across its lanes)
    float yh[C], yl[C];
    {
        // amax in [2^e, 2^(e+1)); piece grids 2^(e-14) and 2^(e-30): every
        // partial sum of up to 256 pieces is an integer below 2^24 in its
        // grid's unit, hence exact in fp32 (e clamped to the fp16 range: a
        // zero or non-finite row takes y = 0 below)
        const int e = min(max(((__float_as_int(amax) >> 23) & 0xff) - 127, -24), 15);
        const float C0 = __int_as_float(((e + 9 + 127) << 23) | 0x400000);  // 1.5 * 2^(e+9)
        const float C1 = __int_as_float(((e - 7 + 127) << 23) | 0x400000);  // 1.5 * 2^(e-7)
        float ph[C], pm[C], pl[C];
#pragma unroll
        for (int j = 0; j < C; ++j) {
            ph[j] = __fsub_rn(__fadd_rn(x[j], C0), C0);
            const float r1 = __fsub_rn(x[j], ph[j]);
            pm[j] = __fsub_rn(__fadd_rn(r1, C1), C1);
            pl[j] = __fsub_rn(r1, pm[j]);
        }
        gen_wht<C, LPR>(ph, ll);
        gen_wht<C, LPR>(pm, ll);
        gen_wht<C, LPR>(pl, ll);
        // den = n sqrt(D) as a double-float
        constexpr int K = log2_d<D>();
        const float p2 = (float)(1 << (K >> 1));
        float dh = nh * p2, dl = nl * p2;
        if (K & 1) {
            const float th = __fmul_rn(dh, SQRT2_HI);
            const float tl = __fadd_rn(__fmaf_rn(dh, SQRT2_HI, -th), __fadd_rn(__fmul_rn(dh, SQRT2_LO), __fmul_rn(dl, SQRT2_HI)));
            fast_two_sum(th, tl, dh, dl);
        }
#pragma unroll
        for (int j = 0; j < C; ++j) {
            float sh, sl;
            two_sum(ph[j], pm[j], sh, sl);
            sl = __fadd_rn(sl, pl[j]);
            fast_two_sum(sh, sl, sh, sl);
            // y = s / den: quotient, exact remainder by FMA, correction
            const float qh = __fdiv_rn(sh, dh);
            const float rem = __fadd_rn(__fadd_rn(__fmaf_rn(-qh, dh, sh), sl), -__fmul_rn(qh, dl));
            fast_two_sum(qh, __fdiv_rn(rem, dh), yh[j], yl[j]);
        }
    }
    if (!(nh > 0.0f) || !(amax <= 65504.0f)) {
        // a zero row has y = 0 (a non-finite one too: any codes are allowed)
#pragma unroll
        for (int j = 0; j < C; ++j) yh[j] = yl[j] = 0.0f;
    }
#pragma unroll
    for (int j = 0; j < C; ++j) {
        const int i1 = gen_count_df<BITS>(bk.b1, yh[j], yl[j]);
        float rh, rl;
        two_sum(yh[j], -bk.c1[i1], rh, rl);
        rl = __fadd_rn(rl, yl[j]);
        fast_two_sum(rh, rl, rh, rl);
        q1[j] = (uint32_t)i1;
        q2[j] = (uint32_t)gen_count_df<BITS>(bk.b2, rh, rl);
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

__device__ __forceinline__ void load8_halves(const __half *src, float (&x)[8])
{
    const uint4 u = *reinterpret_cast<const uint4 *>(src);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w[k]));
        x[2 * k] = f.x;
        x[2 * k + 1] = f.y;
    }
}

__device__ __forceinline__ void load_books(GenBooks &bk, const RvqGenericParams &p, int L)
{
    for (int i = threadIdx.x; i < 17; i += blockDim.x) {
        const float ninf = __int_as_float(0xff800000), pinf = __int_as_float(0x7f800000);
        bk.b1[i] = i == 0 ? ninf : i < L ? p.b1[i - 1] : pinf;
        bk.b2[i] = i == 0 ? ninf : i < L ? p.b2[i - 1] : pinf;
        if (i < 16) bk.c1[i] = p.c1[i];
    }
    __syncthreads();
}

template <int D, int BITS>
__global__ void __launch_bounds__(GEN_WARPS * 32) rvq_generic_encode_kernel(const __grid_constant__ RvqGenericParams p)
{
    using S = GenShape<D>;
    constexpr int LPR = S::LPR, C = S::C, RPW = S::RPW;
    constexpr int E = 32 / BITS;
    constexpr int W = (D + E - 1) / E;
    __shared__ GenBooks bk;
    __shared__ __align__(16) uint8_t cbuf[GEN_WARPS][2][32 * C];
    load_books(bk, p, 1 << BITS);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rl = lane / LPR, ll = lane % LPR;
    const float inv_scale = sqrt_d_f<D>();
    const int nsteps = (p.N + RPW - 1) / RPW;
    for (int step = blockIdx.x * GEN_WARPS + warp; step < nsteps; step += gridDim.x * GEN_WARPS) {
        const int row = step * RPW + rl;
        const bool valid = row < p.N;
        float x[C];
        if (valid) {
            load8_halves(static_cast<const __half *>(p.x) + (size_t)row * D + ll * C, x);
        } else {
#pragma unroll
            for (int j = 0; j < C; ++j) x[j] = 0.0f;
        }
        // row norm: squares of fp16 values are exact in fp32, summed as a
        // double-float (two_sum), the square root corrected once: the norm is
        // the correctly rounded fp32 of the exact one but for rare ties
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
            gen_wht<C, LPR>(y, ll);
            const float inv = qh > 0.0f ? __frcp_rn(nrm * inv_scale) : 0.0f;
            float m = __int_as_float(0x7f800000);
#pragma unroll
            for (int j = 0; j < C; ++j) gen_quant_fast<BITS>(bk, y[j] * inv, q1[j], q2[j], m);
            const bool flag = valid && (!(m >= p.guard) || !(qh > 0.0f));
            if (__any_sync(FULL_MASK, flag)) gen_exact<D, BITS>(bk, x, nh, nl, ll, q1, q2);
        }

        // pack: codes through shared memory, then lane i < RPW * W assembles
        // word i % W of row i / W of this step, for each stream
        uint32_t c1w = 0u, c2w = 0u;
#pragma unroll
        for (int j = 0; j < C; ++j) {
            c1w |= q1[j] << (4 * (j & 3));
            c2w |= q2[j] << (4 * (j & 3));
            if ((j & 3) == 3) {
                // four codes as bytes
                const uint32_t b1 = (c1w & 0xFu) | ((c1w & 0xF0u) << 4) | ((c1w & 0xF00u) << 8) | ((c1w & 0xF000u) << 12);
                const uint32_t b2 = (c2w & 0xFu) | ((c2w & 0xF0u) << 4) | ((c2w & 0xF00u) << 8) | ((c2w & 0xF000u) << 12);
                *reinterpret_cast<uint32_t *>(&cbuf[warp][0][lane * C + j - 3]) = b1;
                *reinterpret_cast<uint32_t *>(&cbuf[warp][1][lane * C + j - 3]) = b2;
                c1w = c2w = 0u;
            }
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
    // merged table c1[i1] + c2[i2] at index i1 * L + i2
    __shared__ float cc[L * L];
    for (int i = threadIdx.x; i < L * L; i += blockDim.x) cc[i] = __fadd_rn(p.c1[i / L], p.c2[i % L]);
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rl = lane / LPR, ll = lane % LPR;
    const float rsd = __frcp_rn(sqrt_d_f<D>());
    const int nsteps = (p.N + RPW - 1) / RPW;
    // the lane's codes i = 8 ll .. 8 ll + 7 lie in words w0 and w0 + 1 (the
    // second only at b = 3)
    const int w0 = (ll * C) / E;
    const int w1 = min((ll * C + C - 1) / E, W - 1);
    for (int step = blockIdx.x * GEN_WARPS + warp; step < nsteps; step += gridDim.x * GEN_WARPS) {
        const int row = step * RPW + rl;
        const bool valid = row < p.N;  // (every lane takes part in the shuffles)
        const uint32_t *r1 = p.p1 + (size_t)row * W, *r2 = p.p2 + (size_t)row * W;
        uint32_t a0 = 0u, b0 = 0u, a1 = 0u, b1 = 0u;
        if (valid) {
            a0 = __ldg(r1 + w0);
            b0 = __ldg(r2 + w0);
            a1 = w1 != w0 ? __ldg(r1 + w1) : a0;
            b1 = w1 != w0 ? __ldg(r2 + w1) : b0;
        }
        float v[C];
#pragma unroll
        for (int j = 0; j < C; ++j) {
            const int i = ll * C + j;
            const bool hi = i >= (w0 + 1) * E;
            const int sh = (i - (hi ? w0 + 1 : w0) * E) * BITS;
            const uint32_t a = hi ? a1 : a0, b = hi ? b1 : b0;
            v[j] = cc[((a >> sh) & (L - 1)) * L + ((b >> sh) & (L - 1))];
        }
        gen_wht<C, LPR>(v, ll);
        if (!valid) continue;
        const float sc = __ldg(p.norms + row) * rsd;
        uint32_t o[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const __half2 h = __floats2half2_rn(v[2 * k] * sc, v[2 * k + 1] * sc);
            o[k] = *reinterpret_cast<const uint32_t *>(&h);
        }
        *reinterpret_cast<uint4 *>(static_cast<__half *>(p.out) + (size_t)row * D + ll * C) = make_uint4(o[0], o[1], o[2], o[3]);
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
