// api.cpp - the extern "C" entry points of include/vq.h: argument
// validation, codebook tables, launch dispatch.  Host code only.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <cuda_runtime_api.h>
#include <mutex>
#include <utility>
#include <vector>

#include "launch.h"
#include "vq.h"

namespace vq {

bool rvq_codebook_f64(int D, int bits, double *g, double *l, double *beta_out);

namespace {

constexpr int kD = 128;
// Guard band (in units of the rotated, unit-norm coordinate y) around every
// boundary: a row with any y (or stage-2 residual) closer than this to a
// boundary is recomputed in exact / double-float arithmetic.  The fp32 fast
// path's error on y is a few 1e-8 (norm, seven butterfly stages, scaling);
// the band is several times the largest error seen on Gaussian rows with
// 40x outlier channels.
constexpr float kGuard = 2.5e-7f;
// the generic (any width) path's guard band: its fp32 rotation runs up to 8
// butterfly stages at D = 256, and a flagged step costs only a binary64 pass
constexpr float kGuardGeneric = 1e-6f;

// RVQ widths and bit counts (the rvq page tests D = 8 .. 256 and b = 1 .. 4);
// D = 128 with b in {1, 2, 4} has the dedicated kernels.
bool rvq_shape_supported(int D, int bits)
{
    return (D == 8 || D == 16 || D == 32 || D == 64 || D == 128 || D == 256) && bits >= 1 && bits <= 4;
}
bool rvq_fast_shape(int D, int bits) { return D == 128 && bits != 3; }
int rvq_words(int D, int bits) { return (D + 32 / bits - 1) / (32 / bits); }

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool overlap(const void *a, size_t na, const void *b, size_t nb)
{
    if (!a || !b || na == 0 || nb == 0) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

bool finite_sorted(const float *v, int n)
{
    for (int i = 0; i < n; ++i) {
        if (!std::isfinite(v[i])) return false;
        if (i > 0 && !(v[i] > v[i - 1])) return false;
    }
    return true;
}

// centroids c[L] ascending, boundaries b[L-1] strictly between neighbours
bool valid_codebook(const float *c, const float *b, int L)
{
    if (!finite_sorted(c, L) || !finite_sorted(b, L - 1)) return false;
    for (int k = 0; k < L - 1; ++k)
        if (!(c[k] < b[k] && b[k] < c[k + 1])) return false;
    return true;
}

vq_status cuda_status(cudaError_t e) { return e == cudaSuccess ? VQ_OK : VQ_ERR_CUDA; }

// Exactly antisymmetric codebook with its middle boundary at 0.
bool symmetric_codebook(const float *c, const float *b, int L)
{
    for (int k = 0; k < L; ++k)
        if (c[k] != -c[L - 1 - k]) return false;
    for (int k = 0; k < L - 1; ++k)
        if (b[k] != -b[L - 2 - k]) return false;
    return b[L / 2 - 1] == 0.0f;
}

// The randomised-sign rotation's sign words (bit j: coordinate j negated), or
// none; the kernels apply them only when has_sgn is set.
template <class P>
void set_signs(P &p, const uint32_t *signs)
{
    p.has_sgn = 0;
    for (int i = 0; i < 4; ++i) {
        p.sgn[i] = signs ? signs[i] : 0u;
        if (p.sgn[i]) p.has_sgn = 1;
    }
}

}  // namespace

// Quantizer tables derived from an RVQ codebook.  Searching for the grid and
// pair tables costs the host 50-200 us per codebook, more than a whole
// decode-time flush on the GPU, so the tables of the last few codebooks are
// kept (keyed by the exact bits of the four arrays) and a call with the same
// books only copies them.  Shared by all threads under a mutex.
namespace {
struct RvqTableEntry {
    int bits = 0;
    float c1[16], b1[16], c2[16], b2[16];
    int mode = 0;
    GridTable t1, t2;
    PairTable pt;
};
constexpr int kTableSlots = 4;
std::mutex g_table_mu;
RvqTableEntry g_tables[kTableSlots];
int g_table_used = 0, g_table_next = 0;

bool same_books(const RvqTableEntry &e, int bits, const float *c1, const float *b1, const float *c2,
                const float *b2)
{
    const int L = 1 << bits;
    return e.bits == bits && std::memcmp(e.c1, c1, 4 * L) == 0 && std::memcmp(e.c2, c2, 4 * L) == 0 &&
           std::memcmp(e.b1, b1, 4 * (L - 1)) == 0 && std::memcmp(e.b2, b2, 4 * (L - 1)) == 0;
}
}  // namespace

int rvq_quantizer_tables(int bits, const float *c1, const float *b1, const float *c2, const float *b2,
                         float guard, GridTable &t1, GridTable &t2, PairTable &pt)
{
    const int L = 1 << bits;
    {
        std::lock_guard<std::mutex> lock(g_table_mu);
        for (int i = 0; i < g_table_used; ++i) {
            const RvqTableEntry &e = g_tables[i];
            if (same_books(e, bits, c1, b1, c2, b2)) {
                t1 = e.t1;
                t2 = e.t2;
                if (e.mode == RVQ_MODE_PAIR) pt = e.pt;
                return e.mode;
            }
        }
    }
    int mode = RVQ_MODE_PLAIN;
    // (b = 2: the symmetric kernel's boundary tests need B, E < 1/4)
    if (bits <= 2 && symmetric_codebook(c1, b1, L) && symmetric_codebook(c2, b2, L) &&
        (bits == 1 || (b1[L - 2] < 0.25f && b2[L - 2] < 0.25f)))
        mode = RVQ_MODE_SYM;
    else if (build_grid(b1, L - 1, guard, t1) && build_grid(b2, L - 1, guard, t2))
        // the shuffle tables also serve the exact recompute of the pair mode
        mode = bits == 4 && build_pair_table(c1, b1, c2, b2, bits, guard, pt) ? RVQ_MODE_PAIR : RVQ_MODE_GRID;
    std::lock_guard<std::mutex> lock(g_table_mu);
    RvqTableEntry &e = g_tables[g_table_next];
    g_table_next = (g_table_next + 1) % kTableSlots;
    if (g_table_used < kTableSlots) ++g_table_used;
    e.bits = bits;
    std::memcpy(e.c1, c1, 4 * L);
    std::memcpy(e.c2, c2, 4 * L);
    std::memcpy(e.b1, b1, 4 * (L - 1));
    std::memcpy(e.b2, b2, 4 * (L - 1));
    e.mode = mode;
    e.t1 = t1;
    e.t2 = t2;
    if (mode == RVQ_MODE_PAIR) e.pt = pt;
    return mode;
}

int sm_count()
{
    // queried on every call (an attribute read, no synchronisation), so the
    // value always belongs to the device that is current now
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    return n;
}

}  // namespace vq

using namespace vq;

extern "C" {

const char *vq_status_str(int s)
{
    switch (s) {
    case VQ_OK: return "VQ_OK";
    case VQ_ERR_INVALID_ARG: return "VQ_ERR_INVALID_ARG";
    case VQ_ERR_UNSUPPORTED: return "VQ_ERR_UNSUPPORTED";
    case VQ_ERR_MISALIGNED: return "VQ_ERR_MISALIGNED";
    case VQ_ERR_ALIASING: return "VQ_ERR_ALIASING";
    case VQ_ERR_CUDA: return "VQ_ERR_CUDA";
    case VQ_ERR_DEVICE: return "VQ_ERR_DEVICE";
    default: return "VQ_ERR_UNKNOWN";
    }
}

const char *vq_version(void) { return "vqflush 0.1.0 sm_103a"; }

vq_status vq_rvq_codebook(int D, int bits, float *c1, float *b1, float *c2, float *b2)
{
    if (!c1 || !b1 || !c2 || !b2) return VQ_ERR_INVALID_ARG;
    if (D <= 0 || bits < 1 || bits > 4) return VQ_ERR_INVALID_ARG;
    const int L = 1 << bits;
    double g[16], l[16], beta;
    if (!rvq_codebook_f64(D, bits, g, l, &beta)) return VQ_ERR_INVALID_ARG;
    for (int k = 0; k < L; ++k) {
        c1[k] = (float)g[k];
        c2[k] = (float)l[k];
    }
    for (int k = 0; k + 1 < L; ++k) {
        b1[k] = (float)(0.5 * (g[k] + g[k + 1]));
        b2[k] = (float)(0.5 * (l[k] + l[k + 1]));
    }
    return VQ_OK;
}

static vq_status rvq_encode_impl(const void *k_f16, int B, int H, int S, int D, int bits,
                                 const float *c1, const float *b1, const float *c2, const float *b2,
                                 uint32_t *packed1, uint32_t *packed2, float *norms,
                                 const int32_t *dst_off, int S_dst, const uint32_t *signs,
                                 vq_stream_t stream)
{
    if (B < 0 || H < 0 || S < 0) return VQ_ERR_INVALID_ARG;
    if (bits < 1 || bits > 4) return VQ_ERR_INVALID_ARG;
    if (!rvq_shape_supported(D, bits)) return VQ_ERR_UNSUPPORTED;
    if (signs && !rvq_fast_shape(D, bits)) return VQ_ERR_UNSUPPORTED;
    if (!c1 || !b1 || !c2 || !b2) return VQ_ERR_INVALID_ARG;
    const int L = 1 << bits;
    if (!valid_codebook(c1, b1, L) || !valid_codebook(c2, b2, L)) return VQ_ERR_INVALID_ARG;
    if (dst_off == nullptr ? S_dst != S : S_dst < S) return VQ_ERR_INVALID_ARG;
    const long long N = (long long)B * H * S;
    const long long Nd = (long long)B * H * S_dst;
    if (N >= (1LL << 31) || Nd >= (1LL << 31)) return VQ_ERR_UNSUPPORTED;
    if (N == 0) return VQ_OK;
    if (!k_f16 || !packed1 || !packed2 || !norms) return VQ_ERR_INVALID_ARG;
    if (!aligned(k_f16, 16) || !aligned(packed1, 16) || !aligned(packed2, 16) || !aligned(norms, 4) ||
        (dst_off && !aligned(dst_off, 4)))
        return VQ_ERR_MISALIGNED;
    const int W = rvq_words(D, bits);
    const size_t in_b = (size_t)N * D * 2, pk_b = (size_t)Nd * W * 4, n_b = (size_t)Nd * 4;
    if (overlap(k_f16, in_b, packed1, pk_b) || overlap(k_f16, in_b, packed2, pk_b) ||
        overlap(k_f16, in_b, norms, n_b) || overlap(packed1, pk_b, packed2, pk_b) ||
        overlap(packed1, pk_b, norms, n_b) || overlap(packed2, pk_b, norms, n_b) ||
        (dst_off && (overlap(dst_off, (size_t)B * 4, packed1, pk_b) ||
                     overlap(dst_off, (size_t)B * 4, packed2, pk_b) ||
                     overlap(dst_off, (size_t)B * 4, norms, n_b))))
        return VQ_ERR_ALIASING;

    if (!rvq_fast_shape(D, bits)) {
        RvqGenericParams g;
        std::memset(&g, 0, sizeof(g));
        g.x = k_f16;
        g.p1 = packed1;
        g.p2 = packed2;
        g.norms = norms;
        g.dst_off = dst_off;
        g.N = (int)N;
        g.S = S;
        g.H = H;
        g.S_dst = S_dst;
        g.D = D;
        g.guard = kGuardGeneric;
        for (int k = 0; k < 16; ++k) {
            g.c1[k] = k < L ? c1[k] : 0.0f;
            g.c2[k] = k < L ? c2[k] : 0.0f;
            g.b1[k] = k < L - 1 ? b1[k] : INFINITY;
            g.b2[k] = k < L - 1 ? b2[k] : INFINITY;
        }
        return cuda_status(launch_rvq_generic(g, bits, true, reinterpret_cast<cudaStream_t>(stream)));
    }
    RvqEncodeParams p;
    std::memset(&p, 0, sizeof(p));
    p.x = k_f16;
    p.p1 = packed1;
    p.p2 = packed2;
    p.norms = norms;
    p.dst_off = dst_off;
    p.N = (int)N;
    p.S = S;
    p.S_q = S;
    p.H = H;
    p.S_dst = S_dst;
    p.guard = kGuard;
    for (int k = 0; k < 16; ++k) {
        p.c1[k] = k < L ? c1[k] : 0.0f;
        p.c2[k] = k < L ? c2[k] : 0.0f;
        p.b1[k] = k < L - 1 ? b1[k] : INFINITY;
        p.b2[k] = k < L - 1 ? b2[k] : INFINITY;
    }
    const int mode = rvq_quantizer_tables(bits, c1, b1, c2, b2, kGuard, p.t1, p.t2, p.pt);
    p.pt_dev = mode == RVQ_MODE_PAIR ? pair_table_device(p.pt, reinterpret_cast<cudaStream_t>(stream)) : nullptr;
    set_signs(p, signs);
    return cuda_status(launch_rvq_encode(p, bits, mode, reinterpret_cast<cudaStream_t>(stream)));
}

vq_status vq_rvq_encode_pack(const void *k_f16, int B, int H, int S, int D, int bits,
                             const float *c1, const float *b1, const float *c2, const float *b2,
                             uint32_t *packed1, uint32_t *packed2, float *norms,
                             const int32_t *dst_off, int S_dst, vq_stream_t stream)
{
    return rvq_encode_impl(k_f16, B, H, S, D, bits, c1, b1, c2, b2, packed1, packed2, norms, dst_off, S_dst,
                           nullptr, stream);
}

vq_status vq_rvq_encode_pack_rs(const void *k_f16, int B, int H, int S, int D, int bits,
                                const float *c1, const float *b1, const float *c2, const float *b2,
                                uint32_t *packed1, uint32_t *packed2, float *norms,
                                const int32_t *dst_off, int S_dst, const uint32_t *signs,
                                vq_stream_t stream)
{
    if (!signs) return VQ_ERR_INVALID_ARG;
    return rvq_encode_impl(k_f16, B, H, S, D, bits, c1, b1, c2, b2, packed1, packed2, norms, dst_off, S_dst,
                           signs, stream);
}

static vq_status rvq_decode_impl(const uint32_t *packed1, const uint32_t *packed2, const float *norms,
                                 int B, int H, int S, int D, int bits, const float *c1, const float *c2,
                                 void *out_f16, const uint32_t *signs, vq_stream_t stream)
{
    if (B < 0 || H < 0 || S < 0) return VQ_ERR_INVALID_ARG;
    if (bits < 1 || bits > 4) return VQ_ERR_INVALID_ARG;
    if (!rvq_shape_supported(D, bits)) return VQ_ERR_UNSUPPORTED;
    if (signs && !rvq_fast_shape(D, bits)) return VQ_ERR_UNSUPPORTED;
    if (!c1 || !c2) return VQ_ERR_INVALID_ARG;
    const int L = 1 << bits;
    for (int k = 0; k < L; ++k)
        if (!std::isfinite(c1[k]) || !std::isfinite(c2[k])) return VQ_ERR_INVALID_ARG;
    const long long N = (long long)B * H * S;
    if (N >= (1LL << 31)) return VQ_ERR_UNSUPPORTED;
    if (N == 0) return VQ_OK;
    if (!packed1 || !packed2 || !norms || !out_f16) return VQ_ERR_INVALID_ARG;
    if (!aligned(packed1, 16) || !aligned(packed2, 16) || !aligned(norms, 4) || !aligned(out_f16, 16))
        return VQ_ERR_MISALIGNED;
    const int W = rvq_words(D, bits);
    const size_t pk_b = (size_t)N * W * 4, out_b = (size_t)N * D * 2;
    if (overlap(out_f16, out_b, packed1, pk_b) || overlap(out_f16, out_b, packed2, pk_b) ||
        overlap(out_f16, out_b, norms, (size_t)N * 4))
        return VQ_ERR_ALIASING;
    if (!rvq_fast_shape(D, bits)) {
        RvqGenericParams g;
        std::memset(&g, 0, sizeof(g));
        g.p1 = const_cast<uint32_t *>(packed1);
        g.p2 = const_cast<uint32_t *>(packed2);
        g.norms = const_cast<float *>(norms);
        g.out = out_f16;
        g.N = (int)N;
        g.D = D;
        for (int k = 0; k < 16; ++k) {
            g.c1[k] = k < L ? c1[k] : 0.0f;
            g.c2[k] = k < L ? c2[k] : 0.0f;
        }
        return cuda_status(launch_rvq_generic(g, bits, false, reinterpret_cast<cudaStream_t>(stream)));
    }
    RvqDecodeParams p;
    std::memset(&p, 0, sizeof(p));
    p.p1 = packed1;
    p.p2 = packed2;
    p.norms = norms;
    p.out = out_f16;
    p.N = (int)N;
    for (int k = 0; k < 16; ++k) {
        p.c1[k] = k < L ? c1[k] : 0.0f;
        p.c2[k] = k < L ? c2[k] : 0.0f;
    }
    set_signs(p, signs);
    return cuda_status(launch_rvq_decode(p, bits, reinterpret_cast<cudaStream_t>(stream)));
}

vq_status vq_rvq_unpack_dequant(const uint32_t *packed1, const uint32_t *packed2, const float *norms,
                                int B, int H, int S, int D, int bits, const float *c1, const float *c2,
                                void *out_f16, vq_stream_t stream)
{
    return rvq_decode_impl(packed1, packed2, norms, B, H, S, D, bits, c1, c2, out_f16, nullptr, stream);
}

vq_status vq_rvq_unpack_dequant_rs(const uint32_t *packed1, const uint32_t *packed2, const float *norms,
                                   int B, int H, int S, int D, int bits, const float *c1, const float *c2,
                                   const uint32_t *signs, void *out_f16, vq_stream_t stream)
{
    if (!signs) return VQ_ERR_INVALID_ARG;
    return rvq_decode_impl(packed1, packed2, norms, B, H, S, D, bits, c1, c2, out_f16, signs, stream);
}

static size_t attend_ws_bytes(int B, int Hq, int nsplit)
{
    return nsplit > 1 ? (size_t)B * Hq * nsplit * AT_PART * sizeof(float) : 0;
}

static vq_status attend_shape_check(int B, int Hq, int Hkv, int S_cap)
{
    if (B < 0 || Hq < 0 || Hkv <= 0 || S_cap < 0) return VQ_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return VQ_ERR_INVALID_ARG;
    const int gq = Hq / Hkv;
    if (Hq > 0 && gq != 1 && gq != 2 && gq != 4 && gq != 8) return VQ_ERR_UNSUPPORTED;
    if ((long long)B * Hkv * S_cap >= (1LL << 31)) return VQ_ERR_UNSUPPORTED;
    return VQ_OK;
}

vq_status vq_rvq_attend_workspace(int B, int Hq, int Hkv, int S_cap, size_t *bytes)
{
    if (!bytes) return VQ_ERR_INVALID_ARG;
    const vq_status st = attend_shape_check(B, Hq, Hkv, S_cap);
    if (st != VQ_OK) return st;
    int nsplit = 1, chunk = 0;
    rvq_attend_plan(B, Hkv, S_cap, &nsplit, &chunk);
    *bytes = attend_ws_bytes(B, Hq, nsplit);
    return VQ_OK;
}

// Shared body of vq_rvq_attend (caller workspace) and vq_rvq_attend_noalloc
// (the library's static scratch, which must hold the default plan's partials).
static vq_status rvq_attend_impl(const void *q_f16, const uint32_t *packed1, const uint32_t *packed2,
                                 const float *norms, const void *v_f16, const int32_t *lens, int B,
                                 int Hq, int Hkv, int S_cap, int D, int bits, const float *c1,
                                 const float *c2, float scale, void *out_f16, void *workspace,
                                 size_t workspace_bytes, bool static_scratch, const uint32_t *signs,
                                 vq_stream_t stream)
{
    vq_status st = attend_shape_check(B, Hq, Hkv, S_cap);
    if (st != VQ_OK) return st;
    if (bits == 3 || (D != kD && D > 0)) return VQ_ERR_UNSUPPORTED;
    if (D != kD || (bits != 1 && bits != 2 && bits != 4)) return VQ_ERR_INVALID_ARG;
    if (!c1 || !c2 || !std::isfinite(scale)) return VQ_ERR_INVALID_ARG;
    const int L = 1 << bits;
    for (int k = 0; k < L; ++k)
        if (!std::isfinite(c1[k]) || !std::isfinite(c2[k])) return VQ_ERR_INVALID_ARG;
    if ((long long)B * Hq == 0) return VQ_OK;
    if (!q_f16 || !out_f16) return VQ_ERR_INVALID_ARG;
    const bool cache = S_cap > 0;
    if (cache && (!packed1 || !packed2 || !norms || !v_f16)) return VQ_ERR_INVALID_ARG;
    if (!aligned(q_f16, 16) || !aligned(out_f16, 16) || (lens && !aligned(lens, 4)) ||
        (cache && (!aligned(packed1, 16) || !aligned(packed2, 16) || !aligned(norms, 4) || !aligned(v_f16, 16))) ||
        (workspace && !aligned(workspace, 16)))
        return VQ_ERR_MISALIGNED;
    const int W = D * bits / 32;
    const size_t rows = (size_t)B * Hkv * S_cap;
    const size_t out_b = (size_t)B * Hq * D * 2;
    if (overlap(out_f16, out_b, q_f16, out_b) || (cache && (overlap(out_f16, out_b, packed1, rows * W * 4) ||
                                                            overlap(out_f16, out_b, packed2, rows * W * 4) ||
                                                            overlap(out_f16, out_b, norms, rows * 4) ||
                                                            overlap(out_f16, out_b, v_f16, rows * D * 2))) ||
        (lens && overlap(out_f16, out_b, lens, (size_t)B * 4)) ||
        (workspace && overlap(out_f16, out_b, workspace, workspace_bytes)))
        return VQ_ERR_ALIASING;
    int nsplit = 1, chunk = 0;
    rvq_attend_plan(B, Hkv, S_cap, &nsplit, &chunk);
    if (static_scratch) {
        // the same plan as with a full workspace, or a size-limit error
        if (attend_static_scratch(&workspace, &workspace_bytes) != cudaSuccess) return VQ_ERR_CUDA;
        if (attend_ws_bytes(B, Hq, nsplit) > workspace_bytes) return VQ_ERR_UNSUPPORTED;
    }
    const size_t per_split = (size_t)B * Hq * AT_PART * sizeof(float);
    if (!workspace) workspace_bytes = 0;
    if (nsplit > 1 && workspace_bytes < attend_ws_bytes(B, Hq, nsplit)) {
        const size_t fit = workspace_bytes / per_split;
        rvq_attend_plan_fit(S_cap, fit > (size_t)nsplit ? nsplit : (int)fit, &nsplit, &chunk);
    }
    RvqAttendParams p;
    std::memset(&p, 0, sizeof(p));
    p.q = q_f16;
    p.p1 = packed1;
    p.p2 = packed2;
    p.norms = norms;
    p.v = v_f16;
    p.lens = lens;
    p.out = out_f16;
    p.ws = static_cast<float *>(workspace);
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.S_cap = S_cap;
    p.nsplit = nsplit;
    p.chunk = chunk;
    p.qscale = (float)((double)scale * 1.4426950408889634 / std::sqrt((double)D));
    for (int k = 0; k < 16; ++k) {
        p.c1[k] = k < L ? c1[k] : 0.0f;
        p.c2[k] = k < L ? c2[k] : 0.0f;
    }
    set_signs(p, signs);
    return cuda_status(launch_rvq_attend(p, bits, reinterpret_cast<cudaStream_t>(stream)));
}

vq_status vq_rvq_attend(const void *q_f16, const uint32_t *packed1, const uint32_t *packed2,
                        const float *norms, const void *v_f16, const int32_t *lens, int B, int Hq,
                        int Hkv, int S_cap, int D, int bits, const float *c1, const float *c2,
                        float scale, void *out_f16, void *workspace, size_t workspace_bytes,
                        vq_stream_t stream)
{
    return rvq_attend_impl(q_f16, packed1, packed2, norms, v_f16, lens, B, Hq, Hkv, S_cap, D, bits, c1, c2,
                           scale, out_f16, workspace, workspace_bytes, false, nullptr, stream);
}

vq_status vq_rvq_attend_rs(const void *q_f16, const uint32_t *packed1, const uint32_t *packed2,
                           const float *norms, const void *v_f16, const int32_t *lens, int B, int Hq,
                           int Hkv, int S_cap, int D, int bits, const float *c1, const float *c2,
                           const uint32_t *signs, float scale, void *out_f16, void *workspace,
                           size_t workspace_bytes, vq_stream_t stream)
{
    if (!signs) return VQ_ERR_INVALID_ARG;
    return rvq_attend_impl(q_f16, packed1, packed2, norms, v_f16, lens, B, Hq, Hkv, S_cap, D, bits, c1, c2,
                           scale, out_f16, workspace, workspace_bytes, false, signs, stream);
}

vq_status vq_rvq_attend_noalloc(const void *q_f16, const uint32_t *packed1, const uint32_t *packed2,
                                const float *norms, const void *v_f16, const int32_t *lens, int B,
                                int Hq, int Hkv, int S_cap, int D, int bits, const float *c1,
                                const float *c2, float scale, void *out_f16, vq_stream_t stream)
{
    return rvq_attend_impl(q_f16, packed1, packed2, norms, v_f16, lens, B, Hq, Hkv, S_cap, D, bits, c1, c2,
                           scale, out_f16, nullptr, 0, true, nullptr, stream);
}

static vq_status kivi_attend_check(int B, int Hq, int Hkv, int S_cap, int R, int D, int bits, int group)
{
    vq_status st = attend_shape_check(B, Hq, Hkv, S_cap);
    if (st != VQ_OK) return st;
    if (R < 0) return VQ_ERR_INVALID_ARG;
    if (bits == 3 || (D != kD && D > 0)) return VQ_ERR_UNSUPPORTED;
    if (D != kD || (bits != 1 && bits != 2 && bits != 4)) return VQ_ERR_INVALID_ARG;
    if (group != 32 && group != 64 && group != 128) return VQ_ERR_UNSUPPORTED;
    if (S_cap % group != 0) return VQ_ERR_UNSUPPORTED;  // whole key groups
    if ((long long)B * Hkv * R >= (1LL << 31)) return VQ_ERR_UNSUPPORTED;
    return VQ_OK;
}

vq_status vq_kivi_attend_workspace(int B, int Hq, int Hkv, int S_cap, int R, size_t *bytes)
{
    if (!bytes) return VQ_ERR_INVALID_ARG;
    const vq_status st = attend_shape_check(B, Hq, Hkv, S_cap);
    if (st != VQ_OK) return st;
    if (R < 0) return VQ_ERR_INVALID_ARG;
    int nsplit = 1, chunk = 0;
    rvq_attend_plan(B, Hkv, S_cap, &nsplit, &chunk);
    const int nparts = nsplit + (R > 0 ? 1 : 0);
    *bytes = nparts > 1 ? (size_t)B * Hq * nparts * AT_PART * sizeof(float) : 0;
    return VQ_OK;
}

vq_status vq_kivi_attend(const void *q_f16, const uint32_t *k_packed, const void *k_scale, const void *k_zero,
                         const uint32_t *v_packed, const void *v_scale, const void *v_zero, const void *k_res,
                         const void *v_res, const int32_t *lens, const int32_t *res_lens, int B, int Hq, int Hkv,
                         int S_cap, int R, int D, int bits, int group, float scale, void *out_f16,
                         void *workspace, size_t workspace_bytes, vq_stream_t stream)
{
    vq_status st = kivi_attend_check(B, Hq, Hkv, S_cap, R, D, bits, group);
    if (st != VQ_OK) return st;
    if (!std::isfinite(scale)) return VQ_ERR_INVALID_ARG;
    if ((long long)B * Hq == 0) return VQ_OK;
    if (!q_f16 || !out_f16) return VQ_ERR_INVALID_ARG;
    const bool cache = S_cap > 0, win = R > 0;
    if (cache && (!k_packed || !k_scale || !k_zero || !v_packed || !v_scale || !v_zero)) return VQ_ERR_INVALID_ARG;
    if (win && (!k_res || !v_res)) return VQ_ERR_INVALID_ARG;
    if (!aligned(q_f16, 16) || !aligned(out_f16, 16) || (lens && !aligned(lens, 4)) ||
        (res_lens && !aligned(res_lens, 4)) || (workspace && !aligned(workspace, 16)) ||
        (cache && (!aligned(k_packed, 16) || !aligned(k_scale, 16) || !aligned(k_zero, 16) ||
                   !aligned(v_packed, 16) || !aligned(v_scale, 16) || !aligned(v_zero, 16))) ||
        (win && (!aligned(k_res, 16) || !aligned(v_res, 16))))
        return VQ_ERR_MISALIGNED;
    const int W = D * bits / 32, NG = S_cap / (group > 0 ? group : 1);
    const size_t BH = (size_t)B * Hkv;
    const size_t out_b = (size_t)B * Hq * D * 2;
    const size_t kp_b = BH * NG * (group * bits / 32) * D * 4, ks_b = BH * NG * D * 2;
    const size_t vp_b = BH * S_cap * W * 4, vs_b = BH * S_cap * (D / group) * 2, r_b = BH * R * D * 2;
    if (overlap(out_f16, out_b, q_f16, out_b) ||
        (cache && (overlap(out_f16, out_b, k_packed, kp_b) || overlap(out_f16, out_b, k_scale, ks_b) ||
                   overlap(out_f16, out_b, k_zero, ks_b) || overlap(out_f16, out_b, v_packed, vp_b) ||
                   overlap(out_f16, out_b, v_scale, vs_b) || overlap(out_f16, out_b, v_zero, vs_b))) ||
        (win && (overlap(out_f16, out_b, k_res, r_b) || overlap(out_f16, out_b, v_res, r_b))) ||
        (lens && overlap(out_f16, out_b, lens, (size_t)B * 4)) ||
        (res_lens && overlap(out_f16, out_b, res_lens, (size_t)B * 4)) ||
        (workspace && overlap(out_f16, out_b, workspace, workspace_bytes)))
        return VQ_ERR_ALIASING;
    int nsplit = 1, chunk = 0;
    rvq_attend_plan(B, Hkv, S_cap, &nsplit, &chunk);
    const size_t per_part = (size_t)B * Hq * AT_PART * sizeof(float);
    if (!workspace) workspace_bytes = 0;
    const int extra = win ? 1 : 0;
    if (nsplit + extra > 1 && workspace_bytes < per_part * (size_t)(nsplit + extra)) {
        // fewer chunks fit; the residual window always needs a part of its own
        const size_t fit = workspace_bytes / per_part;
        if (win && fit < 2) return VQ_ERR_INVALID_ARG;
        rvq_attend_plan_fit(S_cap, (int)((fit > (size_t)(nsplit + extra) ? nsplit + extra : fit) - extra),
                            &nsplit, &chunk);
    }
    if (chunk <= 0) chunk = 32;
    KiviAttendParams p;
    std::memset(&p, 0, sizeof(p));
    p.q = q_f16;
    p.kp = k_packed;
    p.ks = k_scale;
    p.kz = k_zero;
    p.vp = v_packed;
    p.vs = v_scale;
    p.vz = v_zero;
    p.kr = k_res;
    p.vr = v_res;
    p.lens = lens;
    p.res_lens = res_lens;
    p.out = out_f16;
    p.ws = static_cast<float *>(workspace);
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.S_cap = S_cap;
    p.R = R;
    p.G = group;
    p.NG = NG;
    p.nsplit = nsplit;
    p.chunk = chunk;
    p.qscale = (float)((double)scale * 1.4426950408889634);
    return cuda_status(launch_kivi_attend(p, bits, reinterpret_cast<cudaStream_t>(stream)));
}

static vq_status kivi_common_check(int B, int H, int D, int bits, int group)
{
    if (B < 0 || H < 0) return VQ_ERR_INVALID_ARG;
    if (bits == 3 || (D != kD && D > 0)) return VQ_ERR_UNSUPPORTED;
    if (D != kD || (bits != 1 && bits != 2 && bits != 4)) return VQ_ERR_INVALID_ARG;
    if (group <= 0 || D % group != 0 || (group * bits) % 32 != 0) return VQ_ERR_INVALID_ARG;
    if (group != 32 && group != 64 && group != 128) return VQ_ERR_UNSUPPORTED;
    return VQ_OK;
}

vq_status vq_kivi_quant_pack(const void *k_f16, const void *v_f16, int B, int H, int S, int D,
                             int bits, int group, int residual_length,
                             uint32_t *k_packed, void *k_scale, void *k_zero,
                             uint32_t *v_packed, void *v_scale, void *v_zero,
                             const int32_t *dst_off, int S_dst, vq_stream_t stream)
{
    vq_status st = kivi_common_check(B, H, D, bits, group);
    if (st != VQ_OK) return st;
    if (S < 0 || residual_length < 0) return VQ_ERR_INVALID_ARG;
    const int S_q = S - residual_length > 0 ? S - residual_length : 0;
    if (dst_off == nullptr ? S_dst != S_q : S_dst < S_q) return VQ_ERR_INVALID_ARG;
    if ((long long)B * H * S >= (1LL << 31) || (long long)B * H * S_dst >= (1LL << 31))
        return VQ_ERR_UNSUPPORTED;
    if (!k_f16 && !v_f16) return VQ_ERR_INVALID_ARG;
    if (k_f16 && (!k_packed || !k_scale || !k_zero)) return VQ_ERR_INVALID_ARG;
    if (v_f16 && (!v_packed || !v_scale || !v_zero)) return VQ_ERR_INVALID_ARG;
    if ((long long)B * H * S_q == 0) return VQ_OK;
    const int NG_dst = (S_dst + group - 1) / group;
    const size_t in_b = (size_t)B * H * S * D * 2;
    const size_t kpk_b = (size_t)B * H * NG_dst * group * bits / 32 * D * 4;
    const size_t ksz_b = (size_t)B * H * NG_dst * D * 2;
    const size_t vpk_b = (size_t)B * H * S_dst * D * bits / 32 * 4;
    const size_t vsz_b = (size_t)B * H * S_dst * (D / group) * 2;
    if ((k_f16 && (!aligned(k_f16, 16) || !aligned(k_packed, 16) || !aligned(k_scale, 8) ||
                   !aligned(k_zero, 8))) ||
        (v_f16 && (!aligned(v_f16, 16) || !aligned(v_packed, 16) || !aligned(v_scale, 2) ||
                   !aligned(v_zero, 2))) ||
        (dst_off && !aligned(dst_off, 4)))
        return VQ_ERR_MISALIGNED;
    const void *outs[6] = {k_f16 ? k_packed : nullptr, k_f16 ? k_scale : nullptr, k_f16 ? k_zero : nullptr,
                           v_f16 ? v_packed : nullptr, v_f16 ? v_scale : nullptr, v_f16 ? v_zero : nullptr};
    const size_t osz[6] = {kpk_b, ksz_b, ksz_b, vpk_b, vsz_b, vsz_b};
    for (int i = 0; i < 6; ++i) {
        if (overlap(outs[i], osz[i], k_f16, in_b) || overlap(outs[i], osz[i], v_f16, in_b) ||
            (dst_off && overlap(outs[i], osz[i], dst_off, (size_t)B * 4)))
            return VQ_ERR_ALIASING;
        for (int j = i + 1; j < 6; ++j)
            if (overlap(outs[i], osz[i], outs[j], osz[j])) return VQ_ERR_ALIASING;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    KiviQuantParams p;
    std::memset(&p, 0, sizeof(p));
    p.dst_off = dst_off;
    p.B = B;
    p.H = H;
    p.S = S;
    p.S_q = S_q;
    p.S_dst = S_dst;
    p.group = group;
    p.NG_dst = NG_dst;
    if (k_f16) {
        p.x = k_f16;
        p.packed = k_packed;
        p.scale = k_scale;
        p.zero = k_zero;
        cudaError_t e = launch_kivi_quant(p, bits, true, s);
        if (e != cudaSuccess) return VQ_ERR_CUDA;
    }
    if (v_f16) {
        p.x = v_f16;
        p.packed = v_packed;
        p.scale = v_scale;
        p.zero = v_zero;
        cudaError_t e = launch_kivi_quant(p, bits, false, s);
        if (e != cudaSuccess) return VQ_ERR_CUDA;
    }
    return VQ_OK;
}

vq_status vq_flush_decode(const void *k_f16, const void *v_f16, int B, int H, int T, int D,
                          int residual_length, const int32_t *dst_off, int S_dst, int rvq_bits,
                          const float *c1, const float *b1, const float *c2, const float *b2,
                          uint32_t *packed1, uint32_t *packed2, float *norms, int kivi_bits, int group,
                          uint32_t *k_packed, void *k_scale, void *k_zero, uint32_t *v_packed,
                          void *v_scale, void *v_zero, void *k_win, void *v_win, const int32_t *win_off,
                          int R_cap, vq_stream_t stream)
{
    if (B < 0 || H < 0 || T < 0 || residual_length < 0 || residual_length > T) return VQ_ERR_INVALID_ARG;
    if (D != kD) return D > 0 ? VQ_ERR_UNSUPPORTED : VQ_ERR_INVALID_ARG;
    const int R = residual_length, S_q = T - R;
    const bool do_rvq = packed1 != nullptr, do_kk = k_packed != nullptr, do_kv = v_packed != nullptr;
    const bool do_win = R > 0 && (k_win != nullptr || v_win != nullptr);
    if (!do_rvq && !do_kk && !do_kv && !do_win) return VQ_ERR_INVALID_ARG;
    if ((do_rvq || do_kk || (do_win && k_win)) && !k_f16) return VQ_ERR_INVALID_ARG;
    if ((do_kv || (do_win && v_win)) && !v_f16) return VQ_ERR_INVALID_ARG;
    if (dst_off == nullptr ? S_dst != S_q : S_dst < S_q) return VQ_ERR_INVALID_ARG;
    if (do_win && R_cap < R) return VQ_ERR_INVALID_ARG;
    const long long rows = (long long)B * H * T;
    if (rows >= (1LL << 31) || (long long)B * H * S_dst >= (1LL << 31) ||
        (do_win && (long long)B * H * R_cap >= (1LL << 31)))
        return VQ_ERR_UNSUPPORTED;

    FlushParams fp;
    std::memset(&fp, 0, sizeof(fp));
    std::vector<std::pair<const void *, size_t>> ins, outs;
    const size_t in_b = (size_t)rows * kD * 2;
    if (k_f16) ins.push_back({k_f16, in_b});
    if (v_f16) ins.push_back({v_f16, in_b});
    if (dst_off) ins.push_back({dst_off, (size_t)B * 4});
    if (win_off) ins.push_back({win_off, (size_t)B * 4});
    if (!aligned(k_f16, 16) || !aligned(v_f16, 16) || !aligned(dst_off, 4) || !aligned(win_off, 4))
        return VQ_ERR_MISALIGNED;
    if (do_rvq) {
        if (rvq_bits != 1 && rvq_bits != 2 && rvq_bits != 4) return VQ_ERR_INVALID_ARG;
        if (!packed2 || !norms || !c1 || !b1 || !c2 || !b2) return VQ_ERR_INVALID_ARG;
        const int L = 1 << rvq_bits;
        if (!valid_codebook(c1, b1, L) || !valid_codebook(c2, b2, L)) return VQ_ERR_INVALID_ARG;
        if (!aligned(packed1, 16) || !aligned(packed2, 16) || !aligned(norms, 4)) return VQ_ERR_MISALIGNED;
        RvqEncodeParams &p = fp.rvq;
        const int mode = rvq_quantizer_tables(rvq_bits, c1, b1, c2, b2, kGuard, p.t1, p.t2, p.pt);
        p.pt_dev = mode == RVQ_MODE_PAIR ? pair_table_device(p.pt, reinterpret_cast<cudaStream_t>(stream)) : nullptr;
        // the fused flush carries the encoders of the symmetric 1/2-bit books
        // and of 4-bit books with a pair table (the library's books)
        if (!((rvq_bits <= 2 && mode == RVQ_MODE_SYM) || (rvq_bits == 4 && mode == RVQ_MODE_PAIR)))
            return VQ_ERR_UNSUPPORTED;
        fp.rvq_kind = rvq_bits;
        p.x = k_f16;
        p.p1 = packed1;
        p.p2 = packed2;
        p.norms = norms;
        p.dst_off = dst_off;
        p.N = (int)rows;
        p.S = T;
        p.S_q = S_q;
        p.H = H;
        p.S_dst = S_dst;
        p.guard = kGuard;
        for (int k = 0; k < 16; ++k) {
            p.c1[k] = k < L ? c1[k] : 0.0f;
            p.c2[k] = k < L ? c2[k] : 0.0f;
            p.b1[k] = k < L - 1 ? b1[k] : INFINITY;
            p.b2[k] = k < L - 1 ? b2[k] : INFINITY;
        }
        const size_t pk_b = (size_t)B * H * S_dst * rvq_words(kD, rvq_bits) * 4;
        outs.push_back({packed1, pk_b});
        outs.push_back({packed2, pk_b});
        outs.push_back({norms, (size_t)B * H * S_dst * 4});
    }
    if (do_kk || do_kv) {
        if (kivi_bits != 2 && kivi_bits != 4) return VQ_ERR_UNSUPPORTED;
        if (group != 32 && group != 64) return VQ_ERR_UNSUPPORTED;
        fp.kbits = kivi_bits;
        KiviQuantParams q;
        std::memset(&q, 0, sizeof(q));
        q.dst_off = dst_off;
        q.B = B;
        q.H = H;
        q.S = T;
        q.S_q = S_q;
        q.S_dst = S_dst;
        q.group = group;
        q.NG_dst = (S_dst + group - 1) / group;
        const size_t kpk_b = (size_t)B * H * q.NG_dst * group * kivi_bits / 32 * kD * 4;
        const size_t ksz_b = (size_t)B * H * q.NG_dst * kD * 2;
        const size_t vpk_b = (size_t)B * H * S_dst * kD * kivi_bits / 32 * 4;
        const size_t vsz_b = (size_t)B * H * S_dst * (kD / group) * 2;
        if (do_kk) {
            if (!k_scale || !k_zero) return VQ_ERR_INVALID_ARG;
            if (!aligned(k_packed, 16) || !aligned(k_scale, 8) || !aligned(k_zero, 8)) return VQ_ERR_MISALIGNED;
            fp.kk = q;
            fp.kk.x = k_f16;
            fp.kk.packed = k_packed;
            fp.kk.scale = k_scale;
            fp.kk.zero = k_zero;
            outs.push_back({k_packed, kpk_b});
            outs.push_back({k_scale, ksz_b});
            outs.push_back({k_zero, ksz_b});
        }
        if (do_kv) {
            if (!v_scale || !v_zero) return VQ_ERR_INVALID_ARG;
            if (!aligned(v_packed, 16) || !aligned(v_scale, 2) || !aligned(v_zero, 2)) return VQ_ERR_MISALIGNED;
            fp.kv = q;
            fp.kv.x = v_f16;
            fp.kv.packed = v_packed;
            fp.kv.scale = v_scale;
            fp.kv.zero = v_zero;
            outs.push_back({v_packed, vpk_b});
            outs.push_back({v_scale, vsz_b});
            outs.push_back({v_zero, vsz_b});
        }
    }
    if (do_win) {
        if (!aligned(k_win, 16) || !aligned(v_win, 16)) return VQ_ERR_MISALIGNED;
        fp.win.k = k_win ? k_f16 : nullptr;
        fp.win.v = v_win ? v_f16 : nullptr;
        fp.win.k_win = k_win;
        fp.win.v_win = v_win;
        fp.win.win_off = win_off;
        fp.win.B = B;
        fp.win.H = H;
        fp.win.T = T;
        fp.win.R = R;
        fp.win.R_cap = R_cap;
        const size_t w_b = (size_t)B * H * R_cap * kD * 2;
        if (k_win) outs.push_back({k_win, w_b});
        if (v_win) outs.push_back({v_win, w_b});
    }
    for (size_t i = 0; i < outs.size(); ++i) {
        for (const auto &in : ins)
            if (overlap(outs[i].first, outs[i].second, in.first, in.second)) return VQ_ERR_ALIASING;
        for (size_t j = i + 1; j < outs.size(); ++j)
            if (overlap(outs[i].first, outs[i].second, outs[j].first, outs[j].second)) return VQ_ERR_ALIASING;
    }
    if (rows == 0) return VQ_OK;
    return cuda_status(launch_flush(fp, reinterpret_cast<cudaStream_t>(stream)));
}

vq_status vq_kivi_unpack_dequant(const uint32_t *k_packed, const void *k_scale, const void *k_zero,
                                 const uint32_t *v_packed, const void *v_scale, const void *v_zero,
                                 int B, int H, int S_q, int D, int bits, int group,
                                 void *k_out_f16, void *v_out_f16, vq_stream_t stream)
{
    vq_status st = kivi_common_check(B, H, D, bits, group);
    if (st != VQ_OK) return st;
    if (S_q < 0) return VQ_ERR_INVALID_ARG;
    if ((long long)B * H * S_q >= (1LL << 31)) return VQ_ERR_UNSUPPORTED;
    const bool dk = k_out_f16 != nullptr, dv = v_out_f16 != nullptr;
    if (!dk && !dv) return VQ_ERR_INVALID_ARG;
    if (dk && (!k_packed || !k_scale || !k_zero)) return VQ_ERR_INVALID_ARG;
    if (dv && (!v_packed || !v_scale || !v_zero)) return VQ_ERR_INVALID_ARG;
    if ((long long)B * H * S_q == 0) return VQ_OK;
    if ((dk && (!aligned(k_packed, 16) || !aligned(k_scale, 8) || !aligned(k_zero, 8) ||
                !aligned(k_out_f16, 8))) ||
        (dv && (!aligned(v_packed, 16) || !aligned(v_scale, 2) || !aligned(v_zero, 2) ||
                !aligned(v_out_f16, 16))))
        return VQ_ERR_MISALIGNED;
    const int NG = (S_q + group - 1) / group;
    const size_t out_b = (size_t)B * H * S_q * D * 2;
    if (dk && (overlap(k_out_f16, out_b, k_packed, (size_t)B * H * NG * group * bits / 32 * D * 4) ||
               overlap(k_out_f16, out_b, k_scale, (size_t)B * H * NG * D * 2) ||
               overlap(k_out_f16, out_b, k_zero, (size_t)B * H * NG * D * 2)))
        return VQ_ERR_ALIASING;
    if (dv && (overlap(v_out_f16, out_b, v_packed, (size_t)B * H * S_q * D * bits / 32 * 4) ||
               overlap(v_out_f16, out_b, v_scale, (size_t)B * H * S_q * (D / group) * 2) ||
               overlap(v_out_f16, out_b, v_zero, (size_t)B * H * S_q * (D / group) * 2)))
        return VQ_ERR_ALIASING;
    if (dk && dv && overlap(k_out_f16, out_b, v_out_f16, out_b)) return VQ_ERR_ALIASING;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    KiviDequantParams p;
    std::memset(&p, 0, sizeof(p));
    p.BH = B * H;
    p.S_q = S_q;
    p.group = group;
    p.NG = NG;
    if (dk) {
        p.packed = k_packed;
        p.scale = k_scale;
        p.zero = k_zero;
        p.out = k_out_f16;
        if (launch_kivi_dequant(p, bits, true, s) != cudaSuccess) return VQ_ERR_CUDA;
    }
    if (dv) {
        p.packed = v_packed;
        p.scale = v_scale;
        p.zero = v_zero;
        p.out = v_out_f16;
        if (launch_kivi_dequant(p, bits, false, s) != cudaSuccess) return VQ_ERR_CUDA;
    }
    return VQ_OK;
}

vq_status vq_qjl_encode(const void *x_f16, int N, int D, const void *s_f16, int m, uint32_t *packed,
                        void *norms_f16, vq_stream_t stream)
{
    if (N < 0 || D <= 0 || m <= 0) return VQ_ERR_INVALID_ARG;
    if (D != 128 || m % 32 != 0 || m > 256) return VQ_ERR_UNSUPPORTED;
    if (N == 0) return VQ_OK;
    if (!x_f16 || !s_f16 || !packed || !norms_f16) return VQ_ERR_INVALID_ARG;
    if (!aligned(x_f16, 16) || !aligned(s_f16, 16) || !aligned(packed, 16) || !aligned(norms_f16, 16))
        return VQ_ERR_MISALIGNED;
    const size_t xb = (size_t)N * D * 2, sb = (size_t)m * D * 2, pb = (size_t)N * (m / 32) * 4, nb = (size_t)N * 2;
    if (overlap(packed, pb, x_f16, xb) || overlap(packed, pb, s_f16, sb) || overlap(norms_f16, nb, x_f16, xb) ||
        overlap(norms_f16, nb, s_f16, sb) || overlap(packed, pb, norms_f16, nb))
        return VQ_ERR_ALIASING;
    QjlEncodeParams p;
    std::memset(&p, 0, sizeof(p));
    p.x = x_f16;
    p.s = s_f16;
    p.packed = packed;
    p.norms = norms_f16;
    p.N = N;
    p.m = m;
    return launch_qjl_encode(p, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? VQ_OK : VQ_ERR_CUDA;
}

vq_status vq_device_error(vq_stream_t stream, int *code_out)
{
    if (!code_out) return VQ_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    unsigned a = 0, b = 0, c = 0, d = 0;
    if (rvq_take_device_error(&a, s) != cudaSuccess) return VQ_ERR_CUDA;
    if (kivi_take_device_error(&b, s) != cudaSuccess) return VQ_ERR_CUDA;
    if (attend_take_device_error(&c, s) != cudaSuccess) return VQ_ERR_CUDA;
    if (kivi_attend_take_device_error(&d, s) != cudaSuccess) return VQ_ERR_CUDA;
    unsigned e = 0, f = 0, g = 0;
    if (gen_take_device_error(&e, s) != cudaSuccess) return VQ_ERR_CUDA;
    if (qjl_take_device_error(&f, s) != cudaSuccess) return VQ_ERR_CUDA;
    if (flush_take_device_error(&g, s) != cudaSuccess) return VQ_ERR_CUDA;
    *code_out = (int)(a | b | c | d | e | f | g);
    return (a | b | c | d | e | f | g) ? VQ_ERR_DEVICE : VQ_OK;
}

}  // extern "C"
