// launch.h - internal interface between the C-ABI front end (api.cpp) and the
// kernel translation units.  Not installed; users include include/vq.h.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime_api.h>

namespace vq {

// Piecewise lookup that turns a scalar quantizer's boundary count into two
// warp-shuffle table reads.  A value v maps to cell
//   g(v) = RN(31 * sat(fma(v, a, bc)))  in [0, 31]
// (computed on the device as two fp32 FMAs; the host builds the tables by
// evaluating the same fp32 map).  Every boundary lies in its own cell, at least
// the guard band away from the cell edges, so for v in cell g
//   #{k : v > b_k} = code[g] + (v > bnd[g]),
// with bnd[g] = -inf for cells that hold no boundary.
struct GridTable {
    float a, bc;
    float bnd[32];
    int code[32];
};

// Both 4-bit stage codes of a coordinate from one lookup.  The pair (i1, i2)
// is a step function of y whose steps are the stage-1 boundaries and, inside
// stage-1 cell k, the stage-2 boundaries shifted by c1[k] (i2 counts
// y - c1[k] > b2_j, i.e. y > c1[k] + b2_j).  The device maps y to one of
// PT_CELLS cells, g(v) = RN((PT_CELLS - 1) sat(fma(v, a, bc))); a table is
// accepted when every boundary has a cell of its own and every value within
// three guard bands of it maps to that same cell (the encoder evaluates the
// map on the unnormalised transform with a per-row slope, whose rounding the
// extra bands absorb).  Entry g: the boundary in the cell (-inf if none) and
// the pairs below / above it, i1 | i2 << 4, in bytes 0 / 1.
constexpr int PT_CELLS = 512;
struct PairTable {
    float a, bc;
    uint2 ent[PT_CELLS];  // x: boundary (fp32 bits), y: pairs
};

// Division by a divisor d fixed for a launch, for numerators 0 <= n < 2^31:
// q = umulhi(n, m) >> s with l = ceil(log2 d), m = ceil(2^(31 + l) / d),
// s = l - 1 (Granlund and Montgomery, "Division by invariant integers using
// multiplication", 1994, Theorem 4.2 with N = 31); d = 1 is flagged and
// passes n through.
struct FastDiv {
    uint32_t m = 1u, s = 0u, one = 1u;
};

inline FastDiv make_fastdiv(uint32_t d)
{
    FastDiv f;
    if (d <= 1u) return f;
    uint32_t l = 0;
    while ((1ull << l) < d) ++l;
    f.m = (uint32_t)(((1ull << (31 + l)) + d - 1) / d);
    f.s = l - 1;
    f.one = 0u;
    return f;
}

#ifdef __CUDACC__
__device__ __forceinline__ int fdiv(const FastDiv &f, int n)
{
    return f.one ? n : (int)(__umulhi((uint32_t)n, f.m) >> f.s);
}
#endif

struct RvqEncodeParams {
    CUtensorMap tmap;    // x as [N rows, 128] fp16, 64 x 32 boxes, 128-byte swizzle (set by the launcher)
    const void *x;       // fp16 [N, 128]
    uint32_t *p1, *p2;   // [B, H, S_dst, W]
    float *norms;        // [B, H, S_dst]
    const int32_t *dst_off;
    int N, S, H, S_dst;
    int S_q;             // tokens [S_q, S) of each (b, h) slice are not encoded (the fused
                         // flush's fp16 window); S_q = S for vq_rvq_encode_pack
    FastDiv divS, divH;  // by S and by H (set by the launcher)
    float guard;         // |y - boundary| below this sends the row to the exact path
    GridTable t1, t2;
    float c1[16], c2[16], b1[16], b2[16];
    uint32_t sgn[4];  // randomised-sign rotation H diag(s): bit j negates coordinate j
    int has_sgn;
    PairTable pt;  // RVQ_MODE_PAIR only
    const uint2 *pt_dev;  // RVQ_MODE_PAIR: the same cells in device memory, or null (read pt)
};

// The pair table's cells in device memory (static slots, one per distinct
// table, never reused; uploaded on `stream` at first use): the kernels read
// them there instead of from the kernel parameters (which are slow to read
// at per-thread addresses).  Null when every slot is taken, or when the table
// is new and `stream` is being captured (the kernel then reads pt itself).
const uint2 *pair_table_device(const PairTable &pt, cudaStream_t stream);

struct RvqDecodeParams {
    CUtensorMap tm1, tm2;  // b >= 2: the packed words as [N rows, W] uint32, 16-row boxes,
                           // 32- or 64-byte swizzle (set by the launcher)
    const uint32_t *p1, *p2;
    const float *norms;
    void *out;           // fp16 [N, 128]
    int N;
    float c1[16], c2[16];
    uint32_t sgn[4];     // inverse of the randomised-sign rotation: diag(s) H
    int has_sgn;
};

struct KiviQuantParams {
    CUtensorMap tmap;    // x as [B*H, S, 128] fp16 (set by the launcher: box and swizzle per kernel)
    const void *x;       // fp16 [B, H, S, D]
    uint32_t *packed;
    void *scale, *zero;  // fp16
    const int32_t *dst_off;
    int B, H, S, S_q, S_dst, group, NG_dst;
    FastDiv divH, divBlk;  // by H, and by blocks (values) or groups (keys) per (b, h) slice (set by the launcher)
};

struct KiviDequantParams {
    const uint32_t *packed;
    const void *scale, *zero;
    void *out;
    int BH, S_q, group, NG;
};

// Decode-time attention over an RVQ key cache (attend.cu).
constexpr int AT_PART = 2 + 128;  // floats of one split's partial: max, sum, output
struct RvqAttendParams {
    CUtensorMap tmv;               // v as [B*Hkv*S_cap, 128] fp16, 64 x 32 boxes, 128-byte swizzle
                                   // (set by the launcher)
    const void *q;                 // fp16 [B, Hq, 128]
    const uint32_t *p1, *p2;       // [B, Hkv, S_cap, W]
    const float *norms;            // [B, Hkv, S_cap]
    const void *v;                 // fp16 [B, Hkv, S_cap, 128]
    const int32_t *lens;           // [B] or null
    void *out;                     // fp16 [B, Hq, 128]
    float *ws;                     // [B, Hq, nsplit, AT_PART] when nsplit > 1
    int B, Hq, Hkv, S_cap;
    int nsplit, chunk;             // chunks per (sequence, kv head) and keys per chunk
    float qscale;                  // softmax scale * log2(e) / sqrt(128)
    float c1[16], c2[16];
    uint32_t sgn[4];               // randomised-sign rotation of the cache (the query is
    int has_sgn;                   // rotated by H diag(s) too)
};
// Chunking of the keys: the default plan, and the finest one that fits
// `max_splits` partials per (sequence, query head) in a workspace.
void rvq_attend_plan(int B, int Hkv, int S_cap, int *nsplit, int *chunk);
void rvq_attend_plan_fit(int S_cap, int max_splits, int *nsplit, int *chunk);
cudaError_t launch_rvq_attend(const RvqAttendParams &p, int bits, cudaStream_t stream);
// Decode-time attention over a KIVI cache (dequantization inside).
struct KiviAttendParams {
    const void *q;                     // fp16 [B, Hq, 128]
    const uint32_t *kp;                // [B, Hkv, NG, G*b/32, 128]
    const void *ks, *kz;               // fp16 [B, Hkv, NG, 128]
    const uint32_t *vp;                // [B, Hkv, S_cap, 128*b/32]
    const void *vs, *vz;               // fp16 [B, Hkv, S_cap, 128/G]
    const void *kr, *vr;               // fp16 [B, Hkv, R, 128] residual window (R > 0)
    const int32_t *lens, *res_lens;    // [B] or null
    void *out;                         // fp16 [B, Hq, 128]
    float *ws;                         // [B, Hq, nsplit + (R > 0), AT_PART] partials
    int B, Hq, Hkv, S_cap, R, G, NG;
    int nsplit, chunk;                 // chunks of the quantized tokens (part nsplit: the window)
    float qscale;                      // softmax scale * log2(e)
};
cudaError_t launch_kivi_attend(const KiviAttendParams &p, int bits, cudaStream_t stream);
cudaError_t kivi_attend_take_device_error(unsigned *bits, cudaStream_t stream);

// TurboQuantRVQ at the other widths and bit counts (D in {8, ..., 256}, b in
// {1, 2, 3, 4}): words per row W = ceil(D / floor(32 / b)).
struct RvqGenericParams {
    const void *x;                 // encode: fp16 [N, D]
    uint32_t *p1, *p2;             // encode: [B, H, S_dst, W]; decode: [N, W]
    float *norms;                  // encode: [B, H, S_dst]; decode: [N]
    void *out;                     // decode: fp16 [N, D]
    const int32_t *dst_off;        // encode only, or null
    int N, S, H, S_dst, D;
    float guard;                   // |value - boundary| below this: binary64 recompute
    float c1[16], c2[16], b1[16], b2[16];
};
cudaError_t launch_rvq_generic(const RvqGenericParams &p, int bits, bool encode, cudaStream_t stream);
cudaError_t gen_take_device_error(unsigned *bits, cudaStream_t stream);
// QJL encode: sign(S x) bits and ||x|| of every key row.
struct QjlEncodeParams {
    CUtensorMap tmx;               // x as [N, 128] fp16, 64 x 16 boxes, 128-byte swizzle (set by the launcher)
    const void *x;                 // fp16 [N, 128]
    const void *s;                 // fp16 [m, 128] sketch
    uint32_t *packed;              // [N, m / 32]
    void *norms;                   // fp16 [N]
    int N, m;
};
cudaError_t launch_qjl_encode(const QjlEncodeParams &p, cudaStream_t stream);
cudaError_t qjl_take_device_error(unsigned *bits, cudaStream_t stream);

// Device address and size of the library's static attention scratch on the
// current device.
cudaError_t attend_static_scratch(void **ptr, size_t *bytes);

// Encoder quantizer variants: plain boundary count (any codebook), shuffle
// tables (GridTable), and the table-free symmetric 1/2-bit quantizer.
enum RvqMode { RVQ_MODE_PLAIN = 0, RVQ_MODE_GRID = 1, RVQ_MODE_SYM = 2, RVQ_MODE_PAIR = 3 };
cudaError_t launch_rvq_encode(const RvqEncodeParams &p, int bits, int mode, cudaStream_t stream);
// Fill the launcher-set fields (fast divisors, tensor map) of encoder and
// KIVI-quantizer parameters; false if the tensor map cannot be encoded.
// box_rows: rows per TMA box of the input (16: the two-threads-per-row
// encoder; 128: the tensor-memory encoder's tiles).
bool prepare_rvq_encode(RvqEncodeParams &p, int box_rows);
bool prepare_kivi_quant(KiviQuantParams &p, bool per_channel);

// Decode-time flush of one layer in one launch (flush.cu): the RVQ encode of
// the new keys, the KIVI quantization of keys and values, and the copy of
// the tokens that stay fp16 into the caller's window buffers, each part on
// its own range of CTAs of one grid.
struct FlushWindowParams {
    const void *k, *v;       // fp16 [B, H, T, 128]: tokens [T - R, T) are copied
    void *k_win, *v_win;     // fp16 [B, H, R_cap, 128] (either may be null)
    const int32_t *win_off;  // [B] first window row written (null: 0)
    int B, H, T, R, R_cap;
};
struct FlushParams {
    RvqEncodeParams rvq;     // the keys' RVQ part (rvq_kind != 0)
    KiviQuantParams kk, kv;  // KIVI keys / values (x == nullptr: absent)
    FlushWindowParams win;
    int rvq_kind;            // 0: none; 1: symmetric b = 1 books (16-row blocks); 2, 4: the
                             // tensor-memory encoder (symmetric b = 2, b = 4 pair table)
    int kbits;               // KIVI bits (2 or 4; group 32 or 64) when kk or kv is present
    int n_rvq, n_kk, n_kv, n_win;  // CTAs of each part (set by the launcher)
};
cudaError_t launch_flush(FlushParams &p, cudaStream_t stream);
cudaError_t flush_take_device_error(unsigned *bits, cudaStream_t stream);
cudaError_t launch_rvq_decode(const RvqDecodeParams &p, int bits, cudaStream_t stream);
cudaError_t launch_kivi_quant(const KiviQuantParams &p, int bits, bool per_channel,
                              cudaStream_t stream);
cudaError_t launch_kivi_dequant(const KiviDequantParams &p, int bits, bool per_channel,
                                cudaStream_t stream);

// Read and clear the device error word of each kernel unit (bitwise OR).
cudaError_t rvq_take_device_error(unsigned *bits, cudaStream_t stream);
cudaError_t kivi_take_device_error(unsigned *bits, cudaStream_t stream);
cudaError_t attend_take_device_error(unsigned *bits, cudaStream_t stream);

// Host side of the cell map (bit-exact copy of the device's) and the table
// builder; build_grid returns false when no table meets the guard band.
int grid_cell_host(float v, float a, float bc);
bool build_grid(const float *b, int nb, float guard, GridTable &t);
int pair_cell_host(float v, float a, float bc);
bool build_pair_table(const float *c1, const float *b1, const float *c2, const float *b2, int bits,
                      float guard, PairTable &t);

// Number of SMs of the current device.
int sm_count();

// Tiled tensor map of an fp16 tensor: dims innermost first, strides in bytes
// of dims 1..rank-1, box in elements; L2 promotion of 256 bytes when both
// 128-byte halves of a row are loaded together, else 128; false if the
// encoder is unavailable or rejects the layout.
bool encode_tmap_f16(CUtensorMap *map, const void *base, int rank, const uint64_t *dims,
                     const uint64_t *strides, const uint32_t *box, bool swizzle128, bool promote256);
// Tensor map over packed words [rows, words] uint32 with boxes of
// {words, box_rows}; swizzle_bytes 0, 32 or 64 (the row length in bytes).
bool encode_tmap_words(CUtensorMap *map, const void *base, uint64_t rows, uint32_t words, uint32_t box_rows,
                       int swizzle_bytes);

}  // namespace vq
