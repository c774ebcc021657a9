// flush.cu - the decode-time flush of one layer in one launch, for sm_103a.
//
// A decode step appends a block of T new tokens per sequence; the flush
// quantizes its first T - R tokens into the resident caches at each
// sequence's offset and leaves the last R in fp16 (the KIVI residual window:
// kivi page, second post, "What KIVI is"; "Why it's invisible, and why that
// was predictable" names these small flushes as the latency-bound case).
// Done as separate calls, the flush is three or four launches of a few
// microseconds each, every one paying its launch latency, ramp and tail.
// Here one grid does all of it: its CTAs are split into ranges, one per part
// (RVQ encode of the keys, KIVI keys, KIVI values, window copy), sized by
// the part's bytes, and each range runs that part's persistent body (the same
// device code as the stand-alone kernels: rvq_encode.cuh, kivi_quant.cuh)
// over its own items, so the parts overlap on different SMs.  Outputs are
// bit-identical to the stand-alone calls.
#include <cuda_fp16.h>

#include "device_common.cuh"
#include "launch.h"

namespace vq {
VQ_DEFINE_ERROR_WORD(g_flush_err);
}  // namespace vq

#define VQ_RVQ_ERR g_flush_err
#define VQ_KIVI_ERR g_flush_err
#include "kivi_quant.cuh"
#include "rvq_encode.cuh"

namespace vq {

namespace {

constexpr int FL_WARPS = 16;
static_assert(enc_warps(1, MODE_SYM) == FL_WARPS && TE_THREADS == FL_WARPS * 32, "encoder bodies take 16 warps");
static_assert(key_warps<2, 32>() == FL_WARPS && key_warps<4, 64>() == FL_WARPS, "key bodies run 16 warps");

constexpr int WIN_ROWS = 16;  // window rows per warp item

// The window copy: items are (tensor, (b, h), 16-row block of the R window
// tokens); a warp moves one item, 16 B per lane and row chunk, all eight
// loads in flight before the stores.
__device__ __forceinline__ void window_body(const FlushWindowParams &w, int cta, int ncta)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nb = (w.R + WIN_ROWS - 1) / WIN_ROWS;
    const int per_t = w.B * w.H * nb;
    for (int it = cta * FL_WARPS + warp; it < 2 * per_t; it += ncta * FL_WARPS) {
        const int t = it / per_t, r = it - t * per_t;
        const int bh = r / nb, blk = r - bh * nb;
        const uint4 *src = static_cast<const uint4 *>(t ? w.v : w.k);
        uint4 *dst = static_cast<uint4 *>(t ? w.v_win : w.k_win);
        if (src == nullptr || dst == nullptr) continue;
        const int b = bh / w.H;
        const int off = w.win_off ? __ldg(w.win_off + b) : 0;
        if (off < 0 || off > w.R_cap - w.R) {
            if (lane == 0) atomicOr(&g_flush_err, (unsigned)VQ_DEVERR_BAD_OFFSET);
            continue;
        }
        uint4 v[8];
        // 16 rows x 16 chunks of 16 bytes: chunk id = lane + 32 k
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int id = lane + 32 * k, j = blk * WIN_ROWS + (id >> 4);
            if (j < w.R) v[k] = __ldg(src + ((size_t)bh * w.T + (w.T - w.R) + j) * 16 + (id & 15));
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int id = lane + 32 * k, j = blk * WIN_ROWS + (id >> 4);
            if (j < w.R) dst[((size_t)bh * w.R_cap + off + j) * 16 + (id & 15)] = v[k];
        }
    }
}

// Each part is its own function (not inlined), so that the register
// allocation of one part does not weigh on the others.
__device__ __noinline__ void part_rvq1(const RvqEncodeParams &q, int c, int n)
{
    rvq_encode_body<1, MODE_SYM, false>(q, c, n);
}

// the tensor-memory encoder runs all 16 warps of the CTA (two of them fixup warps)
template <int MODE>
__device__ __noinline__ void part_rvq_tm(const RvqEncodeParams &q, int c, int n)
{
    rvq_encode_tm_body<MODE>(q, c, n);
}

__device__ __forceinline__ void part_rvq(const FlushParams &p, int c)
{
    switch (p.rvq_kind) {
    case 1: part_rvq1(p.rvq, c, p.n_rvq); break;
    case 2: part_rvq_tm<MODE_SYM>(p.rvq, c, p.n_rvq); break;
    default: part_rvq_tm<MODE_PAIR>(p.rvq, c, p.n_rvq); break;
    }
}

template <int BITS, int G>
__device__ __noinline__ void part_keys(const KiviQuantParams &q, int c, int n)
{
    kivi_keys_body<BITS, G, FL_WARPS>(q, c, n);
}

template <int BITS, int G>
__device__ __noinline__ void part_values(const KiviQuantParams &q, int c, int n)
{
    kivi_values_body<BITS, G, FL_WARPS>(q, c, n);
}

template <bool KEYS>
__device__ __forceinline__ void kivi_part(const KiviQuantParams &q, int kbits, int cta, int ncta)
{
    const int sel = (kbits == 4 ? 2 : 0) + (q.group == 64 ? 1 : 0);
    if constexpr (KEYS) {
        switch (sel) {
        case 0: part_keys<2, 32>(q, cta, ncta); break;
        case 1: part_keys<2, 64>(q, cta, ncta); break;
        case 2: part_keys<4, 32>(q, cta, ncta); break;
        default: part_keys<4, 64>(q, cta, ncta); break;
        }
    } else {
        switch (sel) {
        case 0: part_values<2, 32>(q, cta, ncta); break;
        case 1: part_values<2, 64>(q, cta, ncta); break;
        case 2: part_values<4, 32>(q, cta, ncta); break;
        default: part_values<4, 64>(q, cta, ncta); break;
        }
    }
}

__global__ void __launch_bounds__(FL_WARPS * 32, 1) vq_flush_kernel(const __grid_constant__ FlushParams p)
{
    int c = blockIdx.x;
    if (c < p.n_rvq) {
        part_rvq(p, c);
        return;
    }
    c -= p.n_rvq;
    if (c < p.n_kk) {
        kivi_part<true>(p.kk, p.kbits, c, p.n_kk);
        return;
    }
    c -= p.n_kk;
    if (c < p.n_kv) {
        kivi_part<false>(p.kv, p.kbits, c, p.n_kv);
        return;
    }
    c -= p.n_kv;
    window_body(p.win, c, p.n_win);
}

// dynamic shared memory of each part (the bodies' own layouts)
int rvq_part_smem(int kind)
{
    switch (kind) {
    case 1: return enc_smem(1, MODE_SYM);
    case 2: return te_smem(MODE_SYM);
    default: return te_smem(MODE_PAIR);
    }
}
int keys_part_smem(int G) { return 1024 + FL_WARPS * ((G <= 64 ? 1 : 2) * G * KEY_ROW + 16) + 16; }
int values_part_smem() { return val_smem_w(FL_WARPS); }

}  // namespace

cudaError_t launch_flush(FlushParams &p, cudaStream_t stream)
{
    // work items (16-row blocks, key half-tiles, window blocks) and bytes per part
    const long long rq = p.rvq_kind ? (long long)p.rvq.N : 0;
    const int kb = p.kbits;
    long long items[4] = {0, 0, 0, 0};
    double bytes[4] = {0, 0, 0, 0};
    int smem = 0;
    if (p.rvq_kind && p.rvq.S_q == 0) p.rvq_kind = 0;  // every token stays fp16
    long long rvq_ctas = 0;  // CTAs the RVQ part can use
    if (p.rvq_kind) {
        // the tensor-memory encoder takes 128-row tiles (one CTA each at a
        // time), the b = 1 encoder 16-row blocks (one per warp)
        const int rows_per_item = p.rvq_kind == 1 ? 16 : TE_M;
        if (!prepare_rvq_encode(p.rvq, rows_per_item)) return cudaErrorInvalidValue;
        items[0] = (rq + rows_per_item - 1) / rows_per_item;
        rvq_ctas = p.rvq_kind == 1 ? (items[0] + FL_WARPS - 1) / FL_WARPS : items[0];
        const long long rows_q = (long long)p.rvq.N / p.rvq.S * p.rvq.S_q;
        bytes[0] = (double)rows_q * (256 + 2 * 16 * p.rvq_kind + 4);
        smem = rvq_part_smem(p.rvq_kind);
    }
    const int G = p.kk.x ? p.kk.group : p.kv.group;
    if (p.kk.x) {
        if (!prepare_kivi_quant(p.kk, true)) return cudaErrorInvalidValue;
        const long long ng = (long long)p.kk.B * p.kk.H * ((p.kk.S_q + G - 1) / G);
        items[1] = 2 * ng;
        bytes[1] = (double)ng * G * D * (2 + kb / 8.0) + (double)ng * D * 4;
        const int m = keys_part_smem(G);
        smem = smem > m ? smem : m;
    }
    if (p.kv.x) {
        if (!prepare_kivi_quant(p.kv, false)) return cudaErrorInvalidValue;
        const long long rows = (long long)p.kv.B * p.kv.H * p.kv.S_q;
        items[2] = (long long)p.kv.B * p.kv.H * ((p.kv.S_q + 15) / 16);
        bytes[2] = (double)rows * D * (2 + kb / 8.0) + (double)rows * (D / G) * 4;
        const int m = values_part_smem();
        smem = smem > m ? smem : m;
    }
    if (p.win.R > 0 && (p.win.k_win || p.win.v_win)) {
        const long long nb = (long long)p.win.B * p.win.H * ((p.win.R + WIN_ROWS - 1) / WIN_ROWS);
        items[3] = 2 * nb;
        bytes[3] = (double)((p.win.k_win ? 1 : 0) + (p.win.v_win ? 1 : 0)) * p.win.B * p.win.H * p.win.R * D * 4;
    }
    // CTAs: at most one per SM in all, shared by each part's expected time:
    // its bytes over the rate one CTA sustains on it (whole-GPU rates in
    // GB/s, measured on a decode flush of 64 sequences x 8 heads x 128 tokens,
    // where each part runs below its full-size rate), at least one per
    // present part and no more than the part has work items for.  The KIVI
    // and window parts balance their items inside each CTA; the RVQ part's
    // CTAs each take whole tiles, so its count is chosen with the others':
    // the split whose slowest part is expected to finish first.
    const double rate[4] = {p.rvq_kind == 4 ? 1300.0 : p.rvq_kind == 2 ? 2800.0 : 2000.0, 4860.0, 3840.0, 6000.0};
    const int sms = sm_count();
    int parts = 0;
    for (int i = 0; i < 4; ++i) parts += items[i] > 0 ? 1 : 0;
    if (parts == 0) return cudaSuccess;
    const int budget = sms > parts ? sms : parts;
    long long useful[4];
    for (int i = 0; i < 4; ++i)
        useful[i] = items[i] == 0 ? 0 : i == 0 ? rvq_ctas : (items[i] + FL_WARPS - 1) / FL_WARPS;
    // the KIVI / window parts share `left` CTAs by their costs; the expected
    // finish (in units of bytes / (GB/s / SM)) of that share
    auto share = [&](int left, int (&n)[4]) {
        double tot = 0.0;
        for (int i = 1; i < 4; ++i)
            if (items[i] > 0) tot += bytes[i] / rate[i];
        double worst = 0.0;
        int used = 0;
        for (int i = 1; i < 4; ++i) {
            n[i] = 0;
            if (items[i] == 0) continue;
            long long w = (long long)(left * (bytes[i] / rate[i]) / tot + 0.5);
            if (w < 1) w = 1;
            if (w > useful[i]) w = useful[i];
            n[i] = (int)w;
            used += n[i];
        }
        while (used > left) {  // rounding overshoot: trim the largest part
            int j = 1;
            for (int i = 2; i < 4; ++i)
                if (n[i] > n[j]) j = i;
            if (n[j] <= 1) break;
            --n[j];
            --used;
        }
        for (int i = 1; i < 4; ++i)
            if (n[i] > 0) {
                const double t = bytes[i] / rate[i] / n[i];
                worst = worst > t ? worst : t;
            }
        return worst;
    };
    int n[4] = {0, 0, 0, 0};
    if (items[0] == 0) {
        (void)share(budget, n);
    } else {
        const int others = parts - 1;
        const double tile_cost = bytes[0] / rate[0] / (double)items[0];  // per item (tile or block)
        const int per_cta = p.rvq_kind == 1 ? FL_WARPS : 1;             // items a CTA takes at once
        double best = 1e300;
        int best_n0 = 1;
        const long long top = useful[0] < budget - others ? useful[0] : budget - others;
        for (int n0 = 1; n0 <= top; ++n0) {
            int m[4];
            const double t_others = others ? share(budget - n0, m) : 0.0;
            const long long waves = (items[0] + (long long)n0 * per_cta - 1) / ((long long)n0 * per_cta);
            const double t0 = waves * per_cta * tile_cost;
            const double t = t0 > t_others ? t0 : t_others;
            if (t < best * (1.0 - 1e-9)) {
                best = t;
                best_n0 = n0;
            }
        }
        n[0] = best_n0;
        if (others) (void)share(budget - best_n0, n);
    }
    int sum = n[0] + n[1] + n[2] + n[3];
    p.n_rvq = n[0];
    p.n_kk = n[1];
    p.n_kv = n[2];
    p.n_win = n[3];
    if (smem < 1024) smem = 1024;
    cudaError_t e = cudaFuncSetAttribute(vq_flush_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    vq_flush_kernel<<<sum, FL_WARPS * 32, smem, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t flush_take_device_error(unsigned *bits, cudaStream_t stream)
{
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(bits, g_flush_err, sizeof(unsigned), 0,
                                              cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    if (*bits) e = cudaMemcpyToSymbolAsync(g_flush_err, &zero, sizeof(unsigned), 0,
                                           cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return e;
    return cudaStreamSynchronize(stream);
}

}  // namespace vq
