/*
 * vq.h - C ABI of the GB300 (sm_103a) KV-cache flush codecs.
 *
 * Two codecs compress fresh fp16 keys/values [B, H, S, D] into bit-packed
 * resident storage and expand it back:
 *
 *   TurboQuantRVQ (VeloxQuant-MLX blog, tag "rvq", sections "The pipeline, as
 *   it actually runs" and "What 'quantize' means here, precisely"): per key
 *   row, L2-normalise (norm kept), rotate by the normalised Walsh-Hadamard
 *   transform y = H u / sqrt(D), quantize y against a Gaussian scalar codebook
 *   by boundary counting (i1 = #{k : y > b1_k}), take the residual
 *   r = y - c1[i1], quantize r against a Laplacian-fit codebook
 *   (i2 = #{k : r > b2_k}), and bit-pack both index streams.
 *
 *   KIVI (VeloxQuant-MLX blog, tag "kivi", first post "What we're actually
 *   optimizing" and second post "What KIVI is"): asymmetric min/max group
 *   quantization, zero = min, scale = (max - min)/(2^b - 1),
 *   q = round_half_even((x - zero)/scale); keys per channel over groups of G
 *   tokens, values per token over groups of G channels; the most recent
 *   residual_length tokens stay fp16 and are not touched.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All tensor pointers are DEVICE pointers unless stated otherwise; fp16
 *    tensors are IEEE binary16 ("void*" in the signatures), row-major and
 *    contiguous.  Codebook arrays are HOST pointers read during the call.
 *  - The caller owns and allocates every buffer.  The library allocates no
 *    memory at call time and never synchronizes with the host.  It keeps
 *    library-wide caches: the quantizer tables of the last four codebooks
 *    (host memory) and, for 16-level books quantized by a pair table (the
 *    library's b = 4 books), that 4 KB table in one of 16 static device slots
 *    per device, uploaded on `stream` by the first call that uses it (a later
 *    call on another stream waits for that upload on the device, if it has
 *    not finished); a call made while `stream` is being captured never
 *    uploads (its kernel then reads the table from its own parameters).
 *  - Work is enqueued on `stream` (NULL = the legacy default stream).
 *  - Arguments are validated on the host before anything is enqueued; a
 *    non-VQ_OK status means nothing was enqueued, except VQ_ERR_CUDA, which
 *    reports a failed launch (the CUDA error is left for the caller to read
 *    with cudaGetLastError()).
 *  - Conditions that depend on device-resident data (destination offsets)
 *    are checked on the device; a violation skips the affected rows and sets
 *    a library-owned device error word, read and cleared by vq_device_error().
 *  - Inputs must be finite; non-finite inputs give unspecified codes but no
 *    out-of-bounds access.
 *  - Packing is LSB first: with E = floor(32/bits) codes per uint32 word,
 *    code j of a word sits at bit shift j*bits.  For bits in {1, 2, 4} these
 *    words have, on a little-endian machine, the same bytes as the byte packer
 *    of the tag "turboquant" page, section "Kernel 1: Bit-Packing".
 *  - Supported: RVQ encode and decode at D in {8, 16, 32, 64, 128, 256} and
 *    bits in {1, 2, 3, 4} (the widths and bit counts the tag "rvq" page tests,
 *    "Bit-exactness, checked the boring way"); D = 128 with bits in {1, 2, 4}
 *    runs the dedicated kernels, the rest a general one.  KIVI, attention and
 *    the randomised-sign calls: D == 128, bits in {1, 2, 4}.
 */
#ifndef VQ_H
#define VQ_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (the same type as cudaStream_t / CUstream). */
typedef struct CUstream_st *vq_stream_t;

typedef enum {
    VQ_OK = 0,
    VQ_ERR_INVALID_ARG = 1,   /* null pointer, bad shape, unsorted codebook ... */
    VQ_ERR_UNSUPPORTED = 2,   /* valid but not implemented (D != 128, bits 3) */
    VQ_ERR_MISALIGNED = 3,    /* a tensor pointer is not 16-byte aligned */
    VQ_ERR_ALIASING = 4,      /* an output overlaps an input or another output */
    VQ_ERR_CUDA = 5,          /* a CUDA launch failed */
    VQ_ERR_DEVICE = 6         /* vq_device_error() found a device-side error */
} vq_status;

/* Device error bits reported by vq_device_error(). */
#define VQ_DEVERR_WAIT_TIMEOUT 0x1 /* a bounded wait on a copy gave up */
#define VQ_DEVERR_BAD_OFFSET 0x2   /* a destination offset was out of range */

/* Human-readable name of a status code (static string). */
const char *vq_status_str(int status);

/* Library version string (static). */
const char *vq_version(void);

/*
 * vq_rvq_codebook - the two TurboQuantRVQ codebooks for head dimension D and
 * `bits` bits per stage, computed on the host in binary64 and rounded to
 * binary32 (VeloxQuant-MLX blog, tag "rvq", "The pipeline, as it actually
 * runs": a Gaussian stage-1 codebook and a Laplacian-fit stage-2 codebook).
 *   c1[2^bits], b1[2^bits - 1]: Lloyd-Max quantizer for N(0, 1/D);
 *   c2[2^bits], b2[2^bits - 1]: Lloyd-Max quantizer for Laplace(0, beta),
 *     beta = E|y - c1[i1(y)]| for y ~ N(0, 1/D) (maximum-likelihood Laplace
 *     scale of the stage-1 residual).
 * Boundaries are midpoints of adjacent centroids.  All four are HOST arrays
 * owned by the caller.  Host only; no GPU needed.
 */
vq_status vq_rvq_codebook(int D, int bits, float *c1, float *b1, float *c2, float *b2);

/*
 * vq_rvq_encode_pack - fused TurboQuantRVQ encode + bit-pack of key rows.
 *   k_f16    [B, H, S, D] fp16, device.
 *   c1, c2   [2^bits] fp32 centroids, host, ascending.
 *   b1, b2   [2^bits - 1] fp32 boundaries, host, strictly increasing, each
 *            strictly between its two neighbouring centroids.
 *   packed1, packed2  [B, H, S_dst, W] uint32, device: the stage-1 and
 *            stage-2 index streams; E = floor(32/bits) codes per word (10 for
 *            bits = 3, whose top two bits stay zero), W = ceil(D/E) words per
 *            row; code of coordinate d in word d/E at shift (d mod E)*bits.
 *   norms    [B, H, S_dst] fp32, device: ||x||_2 of each row.
 *   dst_off  NULL (then S_dst must equal S and rows land at token s) or a
 *            device array [B] of int32 token offsets: row (b, h, s) is written
 *            at token dst_off[b] + s of the destination, which has capacity
 *            S_dst tokens; dst_off[b] + S > S_dst or dst_off[b] < 0 skips
 *            batch b and sets VQ_DEVERR_BAD_OFFSET.
 * A zero row gets norm 0 and the codes of y = 0.  Codes equal those of exact
 * arithmetic; rows with a rotated value within a small guard band of a
 * boundary are recomputed in extended precision on the device.
 */
vq_status vq_rvq_encode_pack(const void *k_f16, int B, int H, int S, int D, int bits,
                             const float *c1, const float *b1, const float *c2, const float *b2,
                             uint32_t *packed1, uint32_t *packed2, float *norms,
                             const int32_t *dst_off, int S_dst, vq_stream_t stream);

/*
 * vq_rvq_unpack_dequant - TurboQuantRVQ unpack + dequant back to keys:
 *   x_hat = n * H (c1[i1] + c2[i2]) / sqrt(D), rounded to fp16.
 * (VeloxQuant-MLX blog, tag "turboquant", "Kernel 5: Fused RVQ Decode +
 * Attend" decodes c1[i1] + c2[i2] in the rotated domain; this call also undoes
 * the rotation, H / sqrt(D) being its own inverse, and re-applies the norm.)
 *   packed1, packed2 [B, H, S, W] uint32 (W as above), norms [B, H, S] fp32, device.
 *   c1, c2 [2^bits] fp32, host.   out_f16 [B, H, S, D] fp16, device.
 */
vq_status vq_rvq_unpack_dequant(const uint32_t *packed1, const uint32_t *packed2,
                                const float *norms, int B, int H, int S, int D, int bits,
                                const float *c1, const float *c2, void *out_f16,
                                vq_stream_t stream);

/*
 * vq_rvq_attend - decode-time attention over a TurboQuantRVQ key cache
 * (VeloxQuant-MLX blog, tag "turboquant", "Kernel 5: Fused RVQ Decode +
 * Attend — Online Softmax Without Materializing K").  For every batch b and
 * query head hq, with kv head h = hq / (Hq / Hkv):
 *   out[b][hq] = sum_s softmax_s(scale * q[b][hq] . k_s) v[b][h][s]
 * over the first lens[b] tokens (all S_cap when lens is NULL; an empty cache
 * gives zeros), where k_s = n_s H (c1[i1] + c2[i2]) / sqrt(D) is the key that
 * vq_rvq_encode_pack encoded.  Keys are scored in the rotated domain straight
 * from their codes and never materialised (fp32 arithmetic).  The weighted
 * sum of the values runs on the tensor cores: fp16 values times each weight
 * carried as two fp16 parts (about 21 bits together), fp32 accumulation.
 * fp16 output.  Rows past lens[b] are never used, whatever they hold.
 *   q [B, Hq, D] fp16, device.
 *   packed1, packed2 [B, Hkv, S_cap, D*bits/32] uint32, norms [B, Hkv, S_cap]
 *     fp32, v [B, Hkv, S_cap, D] fp16, device (an RVQ cache and its values).
 *   lens [B] int32, device, or NULL.   c1, c2 [2^bits] fp32, host.
 *   scale: softmax scale (commonly 1/sqrt(D)).   out [B, Hq, D] fp16, device.
 *   workspace: device memory of at least the size vq_rvq_attend_workspace
 *     reports for these shapes on the current device (NULL when that is 0),
 *     owned by the caller and not shared by calls in flight at the same time;
 *     a smaller workspace is accepted and only reduces the parallelism over
 *     the cache length.
 * D = 128, bits in {1, 2, 4}, Hq = GQ * Hkv with GQ in {1, 2, 4, 8}.
 */
vq_status vq_rvq_attend_workspace(int B, int Hq, int Hkv, int S_cap, size_t *bytes);
vq_status vq_rvq_attend(const void *q_f16, const uint32_t *packed1, const uint32_t *packed2,
                        const float *norms, const void *v_f16, const int32_t *lens, int B, int Hq,
                        int Hkv, int S_cap, int D, int bits, const float *c1, const float *c2,
                        float scale, void *out_f16, void *workspace, size_t workspace_bytes,
                        vq_stream_t stream);

/*
 * vq_rvq_attend_noalloc - vq_rvq_attend without a caller workspace.  The
 * pages have no counterpart to this call: it is a convenience of this
 * library for callers that cannot hand over device memory (for example, a
 * captured graph whose allocations are fixed).  The per-chunk partial
 * results go to a scratch array that the library itself holds in device
 * memory, one per device, VQ_ATTEND_SCRATCH_BYTES long; each call looks up
 * its address on the current device (the first call on a device also loads
 * the library's device code there, so make it before any stream capture).  Same arguments, computation and results
 * as vq_rvq_attend with a workspace of the size vq_rvq_attend_workspace
 * reports (the same chunking, so the output is bit-identical).
 *   Size limit: when that chunking needs more than VQ_ATTEND_SCRATCH_BYTES of
 *     partials (B * Hq * chunks * 520 bytes), the call returns
 *     VQ_ERR_UNSUPPORTED before any launch; use vq_rvq_attend then.
 *   Zero state: nothing in the scratch has to start at zero and the library
 *     never clears it.  Every partial that the combine step reads was written
 *     earlier in the same call by the chunk that owns it; chunks without keys
 *     are neither written nor read, so values left by earlier calls are
 *     never used.
 *   Overlapping calls race: every call on a device shares the one scratch.
 *     Two calls whose kernels can run at the same time (different streams
 *     without an ordering between them, or host threads issuing to different
 *     streams) overwrite each other's partials and give wrong outputs with no
 *     error.  Issue such calls on one stream, or order them with events.
 */
#define VQ_ATTEND_SCRATCH_BYTES (16u * 1024u * 1024u)
vq_status vq_rvq_attend_noalloc(const void *q_f16, const uint32_t *packed1, const uint32_t *packed2,
                                const float *norms, const void *v_f16, const int32_t *lens, int B,
                                int Hq, int Hkv, int S_cap, int D, int bits, const float *c1,
                                const float *c2, float scale, void *out_f16, vq_stream_t stream);

/*
 * Randomised-sign rotation (turboquant page, "Kernel 3: Fused Hadamard +
 * Quantize": TurboQuantMSE's randomized Hadamard preconditioner).  The
 * page's formula reads diag * H * x / sqrt(D) while its kernel flips the
 * signs of x on load and then runs the butterfly; these calls follow the
 * kernel: the rotation is H diag(s) / sqrt(D), with s_j = -1 when bit j of
 * signs[j / 32] is set.  Decode and attention use its transpose
 * diag(s) H / sqrt(D) (keys k = n diag(s) H (c1[i1] + c2[i2]) / sqrt(D); the
 * query is rotated by H diag(s) / sqrt(D)).  signs: host, D/32 uint32 words,
 * chosen by the caller (e.g. from a seed), the same for encode, decode and
 * attention of one cache.  All-zero signs give the plain calls' results bit
 * for bit.  Arguments, layouts and errors otherwise as the plain calls;
 * signs == NULL is VQ_ERR_INVALID_ARG.
 */
vq_status vq_rvq_encode_pack_rs(const void *k_f16, int B, int H, int S, int D, int bits,
                                const float *c1, const float *b1, const float *c2, const float *b2,
                                uint32_t *packed1, uint32_t *packed2, float *norms,
                                const int32_t *dst_off, int S_dst, const uint32_t *signs,
                                vq_stream_t stream);
vq_status vq_rvq_unpack_dequant_rs(const uint32_t *packed1, const uint32_t *packed2, const float *norms,
                                   int B, int H, int S, int D, int bits, const float *c1, const float *c2,
                                   const uint32_t *signs, void *out_f16, vq_stream_t stream);
vq_status vq_rvq_attend_rs(const void *q_f16, const uint32_t *packed1, const uint32_t *packed2,
                           const float *norms, const void *v_f16, const int32_t *lens, int B, int Hq,
                           int Hkv, int S_cap, int D, int bits, const float *c1, const float *c2,
                           const uint32_t *signs, float scale, void *out_f16, void *workspace,
                           size_t workspace_bytes, vq_stream_t stream);

/*
 * vq_kivi_attend - decode-time attention over a KIVI cache, reading the packed
 * codes directly (kivi page, first post, closing section: "Dequant-in-SDPA";
 * the reconstruction is the quantizer's g_hat = q * scale + zero, second
 * post, "What KIVI is").  Keys and values are never reconstructed: with the
 * quantizer's scales and zeros, q . k_t = sum_d (q_d s_d) code + sum_d q_d z_d
 * and sum_t w_t v_t = sum_t (w_t s_t) code + sum_t w_t z_t, and both code sums
 * run on the tensor cores (codes exact in fp16, each float factor carried as
 * two fp16 parts of about 21 bits together, fp32 accumulation); zero terms,
 * softmax and merging are fp32.  Tokens past lens[b] are never used, whatever
 * the cache holds there.
 * For every batch b and query head hq, with kv head h = hq / (Hq / Hkv):
 *   out[b][hq] = sum_t softmax_t(scale * q . k_t) v_t
 * over the first lens[b] quantized tokens (all S_cap when lens is NULL)
 * followed by the first res_lens[b] tokens of the fp16 residual window (all R
 * when res_lens is NULL); an empty cache gives zeros.
 *   q [B, Hq, D] fp16.  Quantized cache, in the layouts vq_kivi_quant_pack
 *   writes with S_dst = S_cap (NG = S_cap / group key groups):
 *     k_packed [B, Hkv, NG, group*bits/32, D] uint32, k_scale, k_zero
 *     [B, Hkv, NG, D] fp16; v_packed [B, Hkv, S_cap, D*bits/32] uint32,
 *     v_scale, v_zero [B, Hkv, S_cap, D/group] fp16.
 *   k_res, v_res [B, Hkv, R, D] fp16 (NULL when R == 0).  All device, 16-byte
 *   aligned.  lens, res_lens [B] int32, device, or NULL.
 *   workspace: as vq_rvq_attend (size from vq_kivi_attend_workspace); with a
 *   residual window at least 2 * B * Hq * 520 bytes are required
 *   (VQ_ERR_INVALID_ARG otherwise).
 * D = 128, bits in {1, 2, 4}, group in {32, 64, 128} with S_cap a multiple of
 * group (VQ_ERR_UNSUPPORTED otherwise), Hq = GQ * Hkv with GQ in {1, 2, 4, 8}.
 */
vq_status vq_kivi_attend_workspace(int B, int Hq, int Hkv, int S_cap, int R, size_t *bytes);
vq_status vq_kivi_attend(const void *q_f16, const uint32_t *k_packed, const void *k_scale,
                         const void *k_zero, const uint32_t *v_packed, const void *v_scale,
                         const void *v_zero, const void *k_res, const void *v_res,
                         const int32_t *lens, const int32_t *res_lens, int B, int Hq, int Hkv,
                         int S_cap, int R, int D, int bits, int group, float scale, void *out_f16,
                         void *workspace, size_t workspace_bytes, vq_stream_t stream);

/*
 * vq_kivi_quant_pack - KIVI flush of K and/or V (either may be NULL, with its
 * outputs).  Quantizes tokens [0, S_q), S_q = S - residual_length; tokens
 * [S_q, S) are the fp16 residual window and are not read or written.
 *   k_f16, v_f16 [B, H, S, D] fp16, device.
 *   group G: G divides D (values); G*bits is a multiple of 32.
 * Key layout (per channel, groups of G tokens; NG = ceil(S_dst/G) groups per
 * (b, h) in the destination):
 *   k_packed [B, H, NG, G*bits/32, D] uint32: word w of group g, channel d
 *     holds tokens g*G + w*E + j at shift j*bits (slots past S_q hold 0);
 *   k_scale, k_zero [B, H, NG, D] fp16.
 * Value layout (per token, groups of G channels):
 *   v_packed [B, H, S_dst, D*bits/32] uint32 (LSB-first along D);
 *   v_scale, v_zero [B, H, S_dst, D/G] fp16.
 * scale = fp16(fp32((max - min)/(2^bits - 1))), zero = min; a constant group
 * stores q = 0 and scale = 0.  Codes use exact arithmetic
 * (t = (x - min)(2^bits - 1)/(max - min), ties to even).
 * dst_off: NULL (S_dst == S_q, token s -> s) or device int32 [B]: token s of
 * batch b lands at dst_off[b] + s; dst_off[b] must be a multiple of G and
 * dst_off[b] + S_q <= S_dst, else batch b is skipped and
 * VQ_DEVERR_BAD_OFFSET is set.  A ragged last key group (S_q mod G != 0) is
 * only supported when it ends the destination sequence.
 */
vq_status vq_kivi_quant_pack(const void *k_f16, const void *v_f16, int B, int H, int S, int D,
                             int bits, int group, int residual_length,
                             uint32_t *k_packed, void *k_scale, void *k_zero,
                             uint32_t *v_packed, void *v_scale, void *v_zero,
                             const int32_t *dst_off, int S_dst, vq_stream_t stream);

/*
 * vq_flush_decode - the decode-time flush of one layer in one launch (kivi
 * page, "Why it's invisible, and why that was predictable": decode flushes are
 * small, so separate launches are mostly latency).  A block of T new tokens
 * per sequence: tokens [0, T - R), R = residual_length, are quantized into
 * the resident caches at the sequences' offsets, tokens [T - R, T) are copied
 * in fp16 into the window buffers.  Every part is optional and equals the
 * stand-alone call bit for bit:
 *   RVQ of the keys (packed1 != NULL; packed2, norms and the four codebook
 *     arrays required): vq_rvq_encode_pack of tokens [0, T - R) with
 *     rvq_bits in {1, 2, 4}; the books must be the library's kind
 *     (symmetric for b = 1, 2, or 16-level books with a pair table, such as
 *     vq_rvq_codebook's), else VQ_ERR_UNSUPPORTED (use vq_rvq_encode_pack);
 *   KIVI of the keys (k_packed != NULL) and of the values (v_packed != NULL):
 *     vq_kivi_quant_pack of tokens [0, T - R) with kivi_bits in {2, 4} and
 *     group in {32, 64} (others: VQ_ERR_UNSUPPORTED);
 *   the window (residual_length > 0, k_win and/or v_win non-NULL): token
 *     T - R + j of (b, h) is copied to row win_off[b] + j of k_win / v_win
 *     [B, H, R_cap, D] fp16 (win_off NULL: row j); win_off[b] + R must not
 *     exceed R_cap, else that batch's window is skipped and
 *     VQ_DEVERR_BAD_OFFSET is set.
 *   k_f16, v_f16 [B, H, T, D] fp16, device (each needed by its parts).
 *   dst_off, S_dst, output layouts and device errors: as vq_rvq_encode_pack
 *     and vq_kivi_quant_pack (S_q = T - R).  D = 128.
 * All pointers are device pointers except the codebooks (host).  Outputs may
 * not overlap each other or the inputs.  Asynchronous on `stream`; one
 * kernel launch; nothing is allocated.
 */
vq_status vq_flush_decode(const void *k_f16, const void *v_f16, int B, int H, int T, int D,
                          int residual_length, const int32_t *dst_off, int S_dst, int rvq_bits,
                          const float *c1, const float *b1, const float *c2, const float *b2,
                          uint32_t *packed1, uint32_t *packed2, float *norms, int kivi_bits, int group,
                          uint32_t *k_packed, void *k_scale, void *k_zero, uint32_t *v_packed,
                          void *v_scale, void *v_zero, void *k_win, void *v_win, const int32_t *win_off,
                          int R_cap, vq_stream_t stream);

/*
 * vq_kivi_unpack_dequant - KIVI unpack + dequant of S_q stored tokens:
 *   x_hat = fp16(q * scale + zero), evaluated exactly and rounded once.
 * Layouts as written by vq_kivi_quant_pack with S_dst = S_q (NG = ceil(S_q/G)).
 * Either side may be NULL.  k_out, v_out [B, H, S_q, D] fp16, device.
 */
vq_status vq_kivi_unpack_dequant(const uint32_t *k_packed, const void *k_scale, const void *k_zero,
                                 const uint32_t *v_packed, const void *v_scale, const void *v_zero,
                                 int B, int H, int S_q, int D, int bits, int group,
                                 void *k_out_f16, void *v_out_f16, vq_stream_t stream);

/*
 * vq_qjl_encode - QJL encode (VeloxQuant-MLX blog, tag "turboquant",
 * "Kernel 4: QJL Encode - Simdgroup Sign Packing"): for every key row x the
 * m bits of sign(S x) - a bit is 1 when the dot product with sketch row j is
 * >= 0 - packed least-significant bit first (bit j of word w is sketch row
 * 32 w + j; on this little-endian device the same bytes as the page's
 * uint8 packing, byte k bit j = row 8 k + j), and ||x|| rounded to fp16.
 * The dot products run on the tensor cores (fp16 products are exact, fp32
 * accumulation): a bit can differ from the exact sign only when |S_j . x| is
 * within about 1e-5 of sum |S_jd x_d|; a norm only when ||x|| is within about
 * 1e-6 (relative) of an fp16 rounding boundary.
 *   x   [N, D] fp16, device (e.g. a key cache [B, H, S, D] as N = B H S rows).
 *   s   [m, D] fp16, device: the sketch matrix (the caller draws it).
 *   packed [N, m / 32] uint32, norms [N] fp16, device.
 * All pointers 16-byte aligned; outputs must not overlap inputs.
 * D = 128, m a multiple of 32 in [32, 256] (VQ_ERR_UNSUPPORTED otherwise).
 * Inputs must be finite.
 */
vq_status vq_qjl_encode(const void *x_f16, int N, int D, const void *s_f16, int m, uint32_t *packed,
                        void *norms_f16, vq_stream_t stream);

/*
 * vq_device_error - waits for `stream`, then reads and clears the library's
 * device error word (VQ_DEVERR_* bits) into *code_out (host pointer).
 * Returns VQ_ERR_DEVICE if the word was non-zero, VQ_OK otherwise.
 */
vq_status vq_device_error(vq_stream_t stream, int *code_out);

#ifdef __cplusplus
}
#endif

#endif /* VQ_H */
