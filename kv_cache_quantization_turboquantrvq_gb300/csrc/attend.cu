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
// Design: one CTA per (batch, kv head, split of the valid tokens), 8 warps;
// the GQ = Hq / Hkv query heads of a kv head are served together, so each key
// and value is read once.  Inside a warp, LK = min(32, 4 GQ) lanes share a
// key, each owning CP = 128 / LK coordinates: the rotated query slices and the
// output accumulators (CP x GQ each) stay in registers, and a key's partial
// dot products are summed over its LK lanes by shuffles.  KP = 32 / LK keys
// run side by side (one per lane group), each group with its own
// online-softmax state, updated four keys at a time.  Groups, then warps, are
// merged at the end.  With several splits the CTA writes its (max, sum,
// unnormalised output) to the caller's workspace and a second kernel
// combines the splits.  Softmax arithmetic is in base 2 (the query carries
// scale * log2(e)).
#include <cuda_fp16.h>

#include "device_common.cuh"
#include "launch.h"

namespace vq {

namespace {

constexpr int D = 128;
constexpr int AT_WARPS = 8;
constexpr int AT_KB = 4;  // keys per lane group per softmax batch
constexpr float NEG_INF = -__builtin_huge_valf();

template <int GQ>
struct AtShape {
    static constexpr int LK = GQ * 4 > 32 ? 32 : (GQ * 4 < 4 ? 4 : GQ * 4);  // lanes per key
    static constexpr int KP = 32 / LK;                                        // keys side by side
    static constexpr int CP = D / LK;                                         // coordinates per lane
    static constexpr int STEP = KP * AT_KB;                                   // keys per warp step
};

__device__ __forceinline__ float exp2_or_zero(float x) { return x == NEG_INF ? 0.0f : exp2f(x); }

// Rotated-domain key values c1[i1] + c2[i2] of CP consecutive coordinates
// whose codes start at bit `sh` of the words w1[0..], w2[0..].
template <int BITS, int CP>
__device__ __forceinline__ void at_decode(const uint32_t *w1, const uint32_t *w2, int sh, float tab,
                                          float tc1, float tc2, float (&y)[CP])
{
    constexpr int E = 32 / BITS;
    if constexpr (BITS == 4) {
#pragma unroll
        for (int c = 0; c < CP; ++c) {
            const int wi = c / E, s = (c % E) * 4 + (CP * BITS < 32 ? sh : 0);
            y[c] = __shfl_sync(FULL_MASK, tc1, (int)(w1[wi] >> s)) + __shfl_sync(FULL_MASK, tc2, (int)(w2[wi] >> s));
        }
    } else {
        // merged index i1 | i2 << BITS: even coordinates from me, odd from mo
        constexpr uint32_t CM = BITS == 2 ? 0x33333333u : 0x55555555u;
        constexpr int NW = (CP * BITS + 31) / 32;
#pragma unroll
        for (int wi = 0; wi < NW; ++wi) {
            uint32_t a = w1[wi], b = w2[wi];
            if constexpr (CP * BITS < 32) {
                a >>= sh;
                b >>= sh;
            }
            const uint32_t me = (a & CM) | ((b << BITS) & ~CM);
            const uint32_t mo = ((a >> BITS) & CM) | (b & ~CM);
            constexpr int PER = CP * BITS < 32 ? CP : E;  // coordinates taken from this word
#pragma unroll
            for (int j = 0; j < PER / 2; ++j) {
                y[wi * E + 2 * j] = __shfl_sync(FULL_MASK, tab, (int)(me >> (2 * BITS * j)));
                y[wi * E + 2 * j + 1] = __shfl_sync(FULL_MASK, tab, (int)(mo >> (2 * BITS * j)));
            }
        }
    }
}

template <int BITS, int GQ>
__global__ void __launch_bounds__(AT_WARPS * 32) rvq_attend_kernel(const __grid_constant__ RvqAttendParams p)
{
    using S = AtShape<GQ>;
    constexpr int LK = S::LK, KP = S::KP, CP = S::CP, STEP = S::STEP;
    constexpr int L = 1 << BITS;
    constexpr int W = D * BITS / 32;
    constexpr int NW = (CP * BITS + 31) / 32;  // code words per lane per key and stream
    __shared__ float qs[GQ][D];
    __shared__ float ms[AT_WARPS][GQ], ls[AT_WARPS][GQ];
    __shared__ float os[AT_WARPS][GQ][D];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int grp = lane / LK, sub = lane % LK;
    const int bh = blockIdx.y, split = blockIdx.x;
    const int b = bh / p.Hkv, h = bh - b * p.Hkv;
    int len = p.lens ? __ldg(p.lens + b) : p.S_cap;
    len = len < 0 ? 0 : (len > p.S_cap ? p.S_cap : len);
    int chunk = (len + p.nsplit - 1) / p.nsplit;
    chunk = (chunk + STEP - 1) / STEP * STEP;
    const int s0 = split * chunk;
    const int s1 = min(len, s0 + chunk);

    // rotated, pre-scaled query of the GQ heads: warp g transforms head g
    if (warp < GQ) {
        const __half *qh = static_cast<const __half *>(p.q) + ((size_t)b * p.Hq + (size_t)h * GQ + warp) * D;
        const uint2 raw = *reinterpret_cast<const uint2 *>(qh + 4 * lane);
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
#pragma unroll
        for (int j = 0; j < 4; ++j) qs[warp][4 * lane + j] = a[j] * p.qscale;
    }
    __syncthreads();
    float qr[GQ][CP];
#pragma unroll
    for (int g = 0; g < GQ; ++g)
#pragma unroll
        for (int c = 0; c < CP; ++c) qr[g][c] = qs[g][sub * CP + c];

    const float tab = BITS == 4 ? 0.0f : p.c1[lane & (L - 1)] + p.c2[(lane >> BITS) & (L - 1)];
    const float tc1 = p.c1[lane & (L - 1)];
    const float tc2 = p.c2[lane & (L - 1)];
    const size_t kbase = (size_t)bh * p.S_cap;
    const int wofs = (sub * CP * BITS) / 32;   // first code word of this lane's coordinates
    const int bsh = (sub * CP * BITS) % 32;    // and their bit offset in it (when CP * BITS < 32)
    const __half *vbase = static_cast<const __half *>(p.v) + kbase * D + sub * CP;

    float m[GQ], l[GQ], o[GQ][CP];
#pragma unroll
    for (int g = 0; g < GQ; ++g) {
        m[g] = NEG_INF;
        l[g] = 0.0f;
#pragma unroll
        for (int c = 0; c < CP; ++c) o[g][c] = 0.0f;
    }

    for (int s = s0 + warp * STEP; s < s1; s += AT_WARPS * STEP) {
        float sc[AT_KB][GQ];
        int kk[AT_KB];
#pragma unroll
        for (int kb = 0; kb < AT_KB; ++kb) {
            const int k = s + kb * KP + grp;
            const bool valid = k < s1;
            kk[kb] = valid ? k : s0;
            const size_t row = kbase + kk[kb];
            uint32_t w1[NW], w2[NW];
#pragma unroll
            for (int i = 0; i < NW; ++i) {
                w1[i] = __ldg(p.p1 + row * W + wofs + i);
                w2[i] = __ldg(p.p2 + row * W + wofs + i);
            }
            const float nrm = __ldg(p.norms + row);
            float y[CP];
            at_decode<BITS, CP>(w1, w2, bsh, tab, tc1, tc2, y);
            float part[GQ];
#pragma unroll
            for (int g = 0; g < GQ; ++g) {
                float acc = 0.0f;
#pragma unroll
                for (int c = 0; c < CP; ++c) acc = fmaf(qr[g][c], y[c], acc);
                part[g] = acc;
            }
#pragma unroll
            for (int off = LK / 2; off >= 1; off >>= 1)
#pragma unroll
                for (int g = 0; g < GQ; ++g) part[g] += __shfl_xor_sync(FULL_MASK, part[g], off);
#pragma unroll
            for (int g = 0; g < GQ; ++g) sc[kb][g] = valid ? part[g] * nrm : NEG_INF;
        }
        // online softmax, one batch of AT_KB keys per lane group; the scores
        // become the batch's weights in place
        float (&w)[AT_KB][GQ] = sc;
#pragma unroll
        for (int g = 0; g < GQ; ++g) {
            float mb = sc[0][g];
#pragma unroll
            for (int kb = 1; kb < AT_KB; ++kb) mb = fmaxf(mb, sc[kb][g]);
            const float mn = fmaxf(m[g], mb);
            const float f = (mn == NEG_INF) ? 1.0f : exp2_or_zero(m[g] == NEG_INF ? NEG_INF : m[g] - mn);
            float sw = 0.0f;
#pragma unroll
            for (int kb = 0; kb < AT_KB; ++kb) {
                w[kb][g] = (sc[kb][g] == NEG_INF) ? 0.0f : exp2f(sc[kb][g] - mn);
                sw += w[kb][g];
            }
            l[g] = l[g] * f + sw;
            m[g] = mn;
#pragma unroll
            for (int c = 0; c < CP; ++c) o[g][c] *= f;
        }
#pragma unroll
        for (int kb = 0; kb < AT_KB; ++kb) {
            float vv[CP];
            const __half *vr = vbase + (size_t)kk[kb] * D;
#pragma unroll
            for (int c = 0; c < CP; c += 8) {
                if constexpr (CP >= 8) {
                    const uint4 u = __ldg(reinterpret_cast<const uint4 *>(vr + c));
                    const __half2 *hh = reinterpret_cast<const __half2 *>(&u);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float2 f2 = __half22float2(hh[j]);
                        vv[c + 2 * j] = f2.x;
                        vv[c + 2 * j + 1] = f2.y;
                    }
                }
            }
            if constexpr (CP == 4) {
                const uint2 u = __ldg(reinterpret_cast<const uint2 *>(vr));
                const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&u.x));
                const float2 bb = __half22float2(*reinterpret_cast<const __half2 *>(&u.y));
                vv[0] = a.x; vv[1] = a.y; vv[2] = bb.x; vv[3] = bb.y;
            }
#pragma unroll
            for (int g = 0; g < GQ; ++g)
#pragma unroll
                for (int c = 0; c < CP; ++c) o[g][c] = fmaf(w[kb][g], vv[c], o[g][c]);
        }
    }

    // merge the KP lane groups of the warp (lanes with the same coordinates)
#pragma unroll
    for (int off = LK; off < 32; off <<= 1) {
#pragma unroll
        for (int g = 0; g < GQ; ++g) {
            const float mo = __shfl_xor_sync(FULL_MASK, m[g], off);
            const float lo = __shfl_xor_sync(FULL_MASK, l[g], off);
            const float mn = fmaxf(m[g], mo);
            const float fa = (m[g] == NEG_INF) ? 0.0f : exp2f(m[g] - mn);
            const float fb = (mo == NEG_INF) ? 0.0f : exp2f(mo - mn);
            l[g] = l[g] * fa + lo * fb;
#pragma unroll
            for (int c = 0; c < CP; ++c) {
                const float oo = __shfl_xor_sync(FULL_MASK, o[g][c], off);
                o[g][c] = o[g][c] * fa + oo * fb;
            }
            m[g] = mn;
        }
    }
    if (grp == 0) {
#pragma unroll
        for (int g = 0; g < GQ; ++g) {
            if (sub == 0) {
                ms[warp][g] = m[g];
                ls[warp][g] = l[g];
            }
#pragma unroll
            for (int c = 0; c < CP; ++c) os[warp][g][sub * CP + c] = o[g][c];
        }
    }
    __syncthreads();

    // merge the warps; write the output (one split) or the partial
    for (int i = threadIdx.x; i < GQ * D; i += blockDim.x) {
        const int g = i / D, d = i - g * D;
        float M = NEG_INF;
#pragma unroll
        for (int k = 0; k < AT_WARPS; ++k) M = fmaxf(M, ms[k][g]);
        float Ls = 0.0f, O = 0.0f;
#pragma unroll
        for (int k = 0; k < AT_WARPS; ++k) {
            const float f = (ms[k][g] == NEG_INF) ? 0.0f : exp2f(ms[k][g] - M);
            Ls = fmaf(ls[k][g], f, Ls);
            O = fmaf(os[k][g][d], f, O);
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

// Combine the splits of one (batch, query head): 128 threads, one per coordinate.
__global__ void __launch_bounds__(D) rvq_attend_combine_kernel(const __grid_constant__ RvqAttendParams p)
{
    const int bq = blockIdx.x, d = threadIdx.x;
    const float *wp = p.ws + (size_t)bq * p.nsplit * AT_PART;
    float M = NEG_INF;
    for (int s = 0; s < p.nsplit; ++s) M = fmaxf(M, wp[(size_t)s * AT_PART]);
    float Ls = 0.0f, O = 0.0f;
    for (int s = 0; s < p.nsplit; ++s) {
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
    dim3 grid(p.nsplit, p.B * p.Hkv);
    rvq_attend_kernel<BITS, GQ><<<grid, AT_WARPS * 32, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || p.nsplit == 1) return e;
    rvq_attend_combine_kernel<<<p.B * p.Hq, D, 0, stream>>>(p);
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

int rvq_attend_splits(int B, int Hkv, int S_cap)
{
    // enough CTAs for two waves over the SMs, but at least one warp step of
    // keys per warp in every split
    const int units = B * Hkv;
    if (units <= 0 || S_cap <= 0) return 1;
    const int want = (2 * sm_count() + units - 1) / units;
    const int most = (S_cap + AT_WARPS * 32 - 1) / (AT_WARPS * 32);
    int n = want < most ? want : most;
    return n < 1 ? 1 : (n > 256 ? 256 : n);
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

}  // namespace vq
