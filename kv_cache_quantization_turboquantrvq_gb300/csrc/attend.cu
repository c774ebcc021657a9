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
// Each warp streams its own tiles of 32 keys: the bulk-copy engine
// (cp.async.bulk) lands the tile's value rows and both code streams - three
// contiguous ranges - in one of two shared-memory stages per warp while the
// warp works on the other.  Per tile:
//   scores   one key per lane: the lane decodes its key's 128 coordinates
//            through a shuffle table (c1 + c2 merged for b <= 2) and forms
//            the GQ dot products with the rotated query, which every lane
//            reads from shared memory as a broadcast (paired-FMA arithmetic);
//   softmax  the tile maximum per head is one warp redux; running maximum,
//            rescale and the per-lane partial sums follow the online softmax;
//   values   lanes own 4 coordinates each; the weights are broadcast from
//            shared memory and the value rows read from the stage.
// Warps, then CTAs (the chunks, through the caller's workspace and a combine
// kernel), are merged at the end.  Softmax arithmetic is in base 2 (the query
// carries scale * log2(e)).
#include <cuda_fp16.h>

#include <mutex>

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
constexpr int TK = 32;  // keys per warp tile: one per lane
constexpr int AT_STAGES = 2;
constexpr float NEG_INF = -__builtin_huge_valf();

template <int BITS>
struct AtTile {
    static constexpr int W = D * BITS / 32;       // code words per key and stream
    static constexpr int VAL = TK * D * 2;        // value rows of a tile (bytes)
    static constexpr int COD = TK * W * 4;        // one code stream of a tile
    static constexpr int STAGE = VAL + 2 * COD;
};

template <int BITS, int GQ>
constexpr int at_smem()
{
    return D * GQ * 4                                  // rotated query [c][g]
           + AT_WARPS * TK * GQ * 4                     // weights [warp][key][g]
           + AT_WARPS * AT_STAGES * AtTile<BITS>::STAGE // stages
           + AT_WARPS * AT_STAGES * 8;                  // mbarriers
}

// Order-preserving map of floats (including -inf) to ints, for a warp redux.
__device__ __forceinline__ int ord_of(float x)
{
    const int i = __float_as_int(x);
    return i >= 0 ? i : i ^ 0x7fffffff;
}
__device__ __forceinline__ float float_of_ord(int i) { return __int_as_float(i >= 0 ? i : i ^ 0x7fffffff); }

__device__ __forceinline__ float2 f2(float a, float b) { return make_float2(a, b); }

// acc[g] += q[c][g] * y for the GQ heads: the rotated query row of coordinate
// c is GQ consecutive floats in shared memory.
template <int GQ>
__device__ __forceinline__ void score_coord(const float *qs, int c, float y, float2 (&acc)[GQ > 1 ? GQ / 2 : 1])
{
    if constexpr (GQ == 2) {
        const float2 q = *reinterpret_cast<const float2 *>(qs + c * 2);
        acc[0] = __ffma2_rn(q, f2(y, y), acc[0]);
    } else if constexpr (GQ >= 4) {
#pragma unroll
        for (int h = 0; h < GQ / 4; ++h) {
            const float4 q = *reinterpret_cast<const float4 *>(qs + c * GQ + 4 * h);
            acc[2 * h] = __ffma2_rn(f2(q.x, q.y), f2(y, y), acc[2 * h]);
            acc[2 * h + 1] = __ffma2_rn(f2(q.z, q.w), f2(y, y), acc[2 * h + 1]);
        }
    }
}

// Dot products of the rotated query with the key whose codes are w1, w2.
// ae/ao take even and odd coordinates (two independent chains).
template <int BITS, int GQ>
__device__ __forceinline__ void key_scores(const float *qs, const uint32_t (&w1)[D * BITS / 32],
                                           const uint32_t (&w2)[D * BITS / 32], float tab, float tc1,
                                           float tc2, float (&s)[GQ])
{
    constexpr int W = D * BITS / 32;
    constexpr int E = 32 / BITS;
    constexpr int NA = GQ > 1 ? GQ / 2 : 1;
    float2 ae[NA], ao[NA];
#pragma unroll
    for (int h = 0; h < NA; ++h) ae[h] = ao[h] = f2(0.0f, 0.0f);
#pragma unroll
    for (int wi = 0; wi < W; ++wi) {
        const uint32_t a = w1[wi], b = w2[wi];
        float y[E];
        if constexpr (BITS == 4) {
#pragma unroll
            for (int c = 0; c < E; ++c)
                y[c] = __shfl_sync(FULL_MASK, tc1, (int)(a >> (4 * c))) +
                       __shfl_sync(FULL_MASK, tc2, (int)(b >> (4 * c)));
        } else {
            // merged index i1 | i2 << BITS: even coordinates from me, odd from mo
            constexpr uint32_t CM = BITS == 2 ? 0x33333333u : 0x55555555u;
            const uint32_t me = (a & CM) | ((b << BITS) & ~CM);
            const uint32_t mo = ((a >> BITS) & CM) | (b & ~CM);
#pragma unroll
            for (int j = 0; j < E / 2; ++j) {
                y[2 * j] = __shfl_sync(FULL_MASK, tab, (int)(me >> (2 * BITS * j)));
                y[2 * j + 1] = __shfl_sync(FULL_MASK, tab, (int)(mo >> (2 * BITS * j)));
            }
        }
        if constexpr (GQ == 1) {
#pragma unroll
            for (int c = 0; c < E; c += 4) {
                const float4 q = *reinterpret_cast<const float4 *>(qs + wi * E + c);
                ae[0] = __ffma2_rn(f2(q.x, q.y), f2(y[c], y[c + 1]), ae[0]);
                ao[0] = __ffma2_rn(f2(q.z, q.w), f2(y[c + 2], y[c + 3]), ao[0]);
            }
        } else {
#pragma unroll
            for (int c = 0; c < E; c += 2) {
                score_coord<GQ>(qs, wi * E + c, y[c], ae);
                score_coord<GQ>(qs, wi * E + c + 1, y[c + 1], ao);
            }
        }
    }
    if constexpr (GQ == 1) {
        s[0] = (ae[0].x + ae[0].y) + (ao[0].x + ao[0].y);
    } else {
#pragma unroll
        for (int h = 0; h < NA; ++h) {
            s[2 * h] = ae[h].x + ao[h].x;
            s[2 * h + 1] = ae[h].y + ao[h].y;
        }
    }
}

template <int BITS, int GQ>
__global__ void __launch_bounds__(AT_WARPS * 32, 1) rvq_attend_kernel(const __grid_constant__ RvqAttendParams p)
{
    using T = AtTile<BITS>;
    constexpr int W = T::W;
    constexpr int L = 1 << BITS;
    extern __shared__ __align__(128) unsigned char smem[];
    float *qs = reinterpret_cast<float *>(smem);
    float *wb = qs + D * GQ;
    unsigned char *stages = reinterpret_cast<unsigned char *>(wb + AT_WARPS * TK * GQ);
    uint64_t *bars = reinterpret_cast<uint64_t *>(stages + AT_WARPS * AT_STAGES * T::STAGE);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.y, split = blockIdx.x;
    const int b = bh / p.Hkv, h = bh - b * p.Hkv;
    int len = p.lens ? __ldg(p.lens + b) : p.S_cap;
    len = len < 0 ? 0 : (len > p.S_cap ? p.S_cap : len);
    const int s0 = split * p.chunk;
    if (s0 >= len && !(split == 0 && p.nsplit == 1)) return;  // no keys: the combine skips this chunk
    const int s1 = min(len, s0 + p.chunk);
    const int ntiles = s1 > s0 ? (s1 - s0 + TK - 1) / TK : 0;

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
            const int k0 = s0 + t * TK;
            const int n = min(TK, s1 - k0);
            unsigned char *dst = my_st + st * T::STAGE;
            mbar_arrive_expect_tx(&my_bar[st], (uint32_t)(n * (D * 2 + 2 * W * 4)));
            bulk_g2s(dst, static_cast<const __half *>(p.v) + (kbase + k0) * D, (uint32_t)(n * D * 2), &my_bar[st], pol);
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
#pragma unroll
        for (int j = 0; j < 4; ++j) qs[(4 * lane + j) * GQ + warp] = a[j] * p.qscale;
    }
    __syncthreads();

    const float tab = BITS == 4 ? 0.0f : p.c1[lane & (L - 1)] + p.c2[(lane >> BITS) & (L - 1)];
    const float tc1 = p.c1[lane & (L - 1)];
    const float tc2 = p.c2[lane & (L - 1)];
    float *my_w = wb + warp * TK * GQ;

    float m[GQ], l[GQ];
    float2 o[GQ][2];  // coordinates 4 lane .. 4 lane + 3
#pragma unroll
    for (int g = 0; g < GQ; ++g) {
        m[g] = NEG_INF;
        l[g] = 0.0f;
        o[g][0] = o[g][1] = f2(0.0f, 0.0f);
    }

    for (int it = 0;; ++it) {
        const int t = warp + it * AT_WARPS;
        if (t >= ntiles) break;
        const int st = it % AT_STAGES;
        const int k0 = s0 + t * TK;
        const int n = min(TK, s1 - k0);
        const bool valid = lane < n;
        const float nrm = valid ? __ldg(p.norms + kbase + k0 + lane) : 0.0f;
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

        // scores: one key per lane
        uint32_t w1[W], w2[W];
        {
            const uint4 *c1p = reinterpret_cast<const uint4 *>(sb + T::VAL) + lane * (W / 4);
            const uint4 *c2p = reinterpret_cast<const uint4 *>(sb + T::VAL + T::COD) + lane * (W / 4);
#pragma unroll
            for (int i = 0; i < W / 4; ++i) {
                const uint4 x = c1p[i], y = c2p[i];
                w1[4 * i] = x.x; w1[4 * i + 1] = x.y; w1[4 * i + 2] = x.z; w1[4 * i + 3] = x.w;
                w2[4 * i] = y.x; w2[4 * i + 1] = y.y; w2[4 * i + 2] = y.z; w2[4 * i + 3] = y.w;
            }
        }
        float s[GQ];
        key_scores<BITS, GQ>(qs, w1, w2, tab, tc1, tc2, s);

        // online softmax over the tile
#pragma unroll
        for (int g = 0; g < GQ; ++g) {
            const float sc = valid ? s[g] * nrm : NEG_INF;
            const float mt = float_of_ord(__reduce_max_sync(FULL_MASK, ord_of(sc)));
            if (mt > m[g]) {  // warp-uniform
                const float f = exp2f(m[g] - mt);
                l[g] *= f;
                o[g][0] = __fmul2_rn(o[g][0], f2(f, f));
                o[g][1] = __fmul2_rn(o[g][1], f2(f, f));
                m[g] = mt;
            }
            const float w = exp2f(sc - m[g]);
            l[g] += w;
            s[g] = w;
        }
        if constexpr (GQ == 1) {
            my_w[lane] = s[0];
        } else if constexpr (GQ == 2) {
            *reinterpret_cast<float2 *>(my_w + lane * 2) = f2(s[0], s[1]);
        } else {
#pragma unroll
            for (int g = 0; g < GQ; g += 4)
                *reinterpret_cast<float4 *>(my_w + lane * GQ + g) = make_float4(s[g], s[g + 1], s[g + 2], s[g + 3]);
        }
        __syncwarp();

        // values: lane owns coordinates 4 lane .. 4 lane + 3
        const uint2 *vr = reinterpret_cast<const uint2 *>(sb) + lane;
        auto accumulate = [&](int k) {
            const uint2 u = vr[k * (D / 4)];
            const float2 v01 = __half22float2(*reinterpret_cast<const __half2 *>(&u.x));
            const float2 v23 = __half22float2(*reinterpret_cast<const __half2 *>(&u.y));
            float wk[GQ];
            if constexpr (GQ == 1) {
                wk[0] = my_w[k];
            } else if constexpr (GQ == 2) {
                const float2 x = *reinterpret_cast<const float2 *>(my_w + k * 2);
                wk[0] = x.x; wk[1] = x.y;
            } else {
#pragma unroll
                for (int g = 0; g < GQ; g += 4) {
                    const float4 x = *reinterpret_cast<const float4 *>(my_w + k * GQ + g);
                    wk[g] = x.x; wk[g + 1] = x.y; wk[g + 2] = x.z; wk[g + 3] = x.w;
                }
            }
#pragma unroll
            for (int g = 0; g < GQ; ++g) {
                o[g][0] = __ffma2_rn(f2(wk[g], wk[g]), v01, o[g][0]);
                o[g][1] = __ffma2_rn(f2(wk[g], wk[g]), v23, o[g][1]);
            }
        };
        if (n == TK) {
#pragma unroll 8
            for (int k = 0; k < TK; ++k) accumulate(k);
        } else {
            for (int k = 0; k < n; ++k) accumulate(k);
        }

        // the stage and the weights are consumed: recycle the stage
        __syncwarp();
        fence_proxy_async_smem();
        if (t + AT_STAGES * AT_WARPS < ntiles) issue(t + AT_STAGES * AT_WARPS, st);
    }

    // per-warp sums, then merge the warps through shared memory (the stages
    // are free: every copy this CTA issued has been waited for)
#pragma unroll
    for (int g = 0; g < GQ; ++g)
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) l[g] += __shfl_xor_sync(FULL_MASK, l[g], off);
    __syncthreads();
    float *ms = reinterpret_cast<float *>(stages);
    float *ls = ms + AT_WARPS * GQ;
    float *os = ls + AT_WARPS * GQ;  // [warp][g][D]
#pragma unroll
    for (int g = 0; g < GQ; ++g) {
        if (lane == 0) {
            ms[warp * GQ + g] = m[g];
            ls[warp * GQ + g] = l[g];
        }
        *reinterpret_cast<float4 *>(os + (warp * GQ + g) * D + 4 * lane) =
            make_float4(o[g][0].x, o[g][0].y, o[g][1].x, o[g][1].y);
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
    auto kern = rvq_attend_kernel<BITS, GQ>;
    constexpr int smem = at_smem<BITS, GQ>();
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    dim3 grid(p.nsplit, p.B * p.Hkv);
    kern<<<grid, AT_WARPS * 32, smem, stream>>>(p);
    e = cudaGetLastError();
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
    // the symbol's device address, looked up once per device
    static std::mutex mu;
    static void *addr[64] = {nullptr};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (addr[dev] == nullptr) {
        e = cudaGetSymbolAddress(&addr[dev], g_at_scratch);
        if (e != cudaSuccess) return e;
    }
    *ptr = addr[dev];
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
