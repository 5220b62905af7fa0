/*
 * tq.h -- C ABI of the rotated + quantized KV-cache library (GB300, sm_103a).
 *
 * The method (web pages on the subject, cited by page title and section):
 *   - "turboquant-mlx" (TurboQuant-MLX v2.0 README), "Walsh-Hadamard Rotation":
 *     each key/value head vector is rotated by the SRHT R = D H D / sqrt(d)
 *     (D a seeded sign diagonal, H the Sylvester Hadamard matrix), O(d log d).
 *   - "TurboMOQ" (turboMOQ README), "Architecture": keys are quantized on a
 *     symmetric grid, values with a Gaussian Lloyd-Max codebook, 1-8 bits per
 *     head, with an optional 1-bit QJL sign sketch of the key residual ("QJL
 *     residual correction (sub-2-bit)"); "Progressive temporal tiering": token
 *     ranges by age carry different bit widths (16 = kept in fp16).
 *   - "turboquant-mlx", "FP16 Attention Sinks" and "Dynamic Chunk Buffering":
 *     the first 128 tokens stay fp16; new tokens are compressed 64 at a time.
 *   - "turboquant-mlx" skill note, "Optimisations Metal": attention runs on the
 *     compressed cache with the inverse transform pulled out of the V sum.
 *
 * Conventions for every entry point:
 *   - Return value: TQ_OK (0) or a negative tq_status.  Arguments are checked on
 *     the host before anything is launched; nothing aborts or throws.
 *   - Device pointers are caller-owned CUDA device memory; the library never
 *     allocates or frees device memory.  Host pointers are caller-owned too.
 *     The one exception on the host: decode calls keep eight pinned host
 *     staging buffers for their plan upload (allocated by the first calls,
 *     grown when a larger plan needs it, kept until the process exits).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Launches are asynchronous on it; errors of kernel execution surface at
 *     the caller's next synchronisation.  TQ_ERR_CUDA reports a launch error
 *     whose cudaError_t value tq_last_cuda_error() returns.
 *   - fp16 data are IEEE binary16 bit patterns (uint16_t / __half).
 *   - Device buffers must be 16-byte aligned (TQ_ERR_ALIGN otherwise).
 *   - head_dim is any power of two from 16 to 1024 ("turboquant-mlx",
 *     "Walsh-Hadamard Rotation": WalshHadamardRotation(head_dim, seed)).  At
 *     head_dim = 128 every call and option below is available (decode with GQA
 *     group sizes 1, 2 and 4, query heads per KV head).  Other head dims take
 *     tq_compress, tq_dequantize and tq_decode_attention (GQA 1 to 4) with the
 *     SRHT rotation and the Gaussian value codebook; QJL sketches (keys or
 *     values), dense rotations, the sphere codebook, attention-mass outputs
 *     and tq_requantize return TQ_ERR_UNSUPPORTED there.
 */
#ifndef TQ_H
#define TQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TQ_MAX_HEADS 16    /* KV heads per layer */
#define TQ_MAX_SEGMENTS 8  /* segments per layer in one decode call */
#define TQ_MAX_HEAD_DIM 1024

typedef int tq_status;
#define TQ_OK 0
#define TQ_ERR_ARG (-1)         /* a NULL / out-of-range argument */
#define TQ_ERR_UNSUPPORTED (-2) /* a valid shape the kernels do not implement */
#define TQ_ERR_ALIGN (-3)       /* a device pointer or stride is not 16-byte aligned */
#define TQ_ERR_SIZE (-4)        /* a buffer is too small (workspace, capacity) */
#define TQ_ERR_CUDA (-5)        /* a CUDA runtime call failed; see tq_last_cuda_error */
#define TQ_ERR_TIMEOUT (-6)     /* a kernel gave up a bounded wait for its own copies
                                   (tq_decode_error_flag, tq_compress_error_flag):
                                   the output of that call is incomplete */

/* Human-readable name of a status.  Never NULL. */
const char *tq_status_string(tq_status s);
/* cudaError_t value of the last TQ_ERR_CUDA returned on this host thread. */
int tq_last_cuda_error(void);
/* Library version, major*10000 + minor*100 + patch. */
int tq_version(void);

/* ------------------------------------------------------------------------ */
/* Rotation ("turboquant-mlx", "Walsh-Hadamard Rotation":                      */
/* WalshHadamardRotation(head_dim, seed)).                                     */
/* ------------------------------------------------------------------------ */
typedef struct {
    int head_dim;          /* d: a power of two, 16..1024 */
    uint64_t seed;         /* layer l conventionally uses seed + l */
    uint32_t sign_bits[TQ_MAX_HEAD_DIM / 32]; /* bit i set <=> D_i = -1 */
    const float *dense;    /* NULL: the SRHT above.  Else a dense rotation
                              ("TurboMOQ", "Stable QR Rotation"): device d x d
                              floats, row-major, orthogonal, y = Q x (caller-owned,
                              16-byte aligned; see tq_make_haar_rotation).  Used
                              by tq_compress (tensor-core kernel, no QJL heads),
                              tq_dequantize and tq_decode_attention. */
} tq_rotation;

/* Fill *rot (caller-owned, plain data) with the sign diagonal of
 * R = D H D / sqrt(d): D_i = -1 iff the top bit of the i-th SplitMix64 output
 * of `seed` is set.  R is symmetric and R R = I.  TQ_ERR_ARG on a NULL rot or a
 * head_dim that is not a power of two in [16, 1024]. */
tq_status tq_make_rotation(int head_dim, uint64_t seed, tq_rotation *rot);

/* Haar-random rotation ("TurboMOQ", "Stable QR Rotation": QR factorisation of
 * a Gaussian matrix): G = the N(0,1) matrix tq_make_qjl(head_dim, head_dim,
 * seed) writes, factored G = Q R by Householder reflections in binary64, the
 * columns of Q multiplied by the signs of diag(R) (so that Q is Haar
 * distributed), rounded to binary32.  Q: host, head_dim^2 floats, row-major.
 * Copy it to the device and set tq_rotation.dense to use it.  TQ_ERR_ARG on a
 * NULL Q or a head_dim that is not a power of two in [16, 1024]. */
tq_status tq_make_haar_rotation(int head_dim, uint64_t seed, float *Q);

/* ------------------------------------------------------------------------ */
/* Value codebook ("TurboMOQ", "Architecture": Lloyd-Max codebook -> grid      */
/* quantize).  Gaussian N(0,1) Lloyd-Max quantizer with 2^bits levels, fitted  */
/* in binary64 by Lloyd's iteration from the quantiles (k + 1/2)/2^bits until   */
/* no level moves by more than 1e-13, then rounded to binary32.  Thresholds are  */
/* midpoints of adjacent levels (the middle one is exactly 0).                 */
/* ------------------------------------------------------------------------ */
/* centroids: 2^bits floats (host); thresholds: 2^bits - 1 floats (host, may be
 * NULL).  Results are cached per bit width after the first call (the 8-bit fit
 * takes about a second).  TQ_ERR_ARG for bits outside 1..8 or NULL centroids. */
tq_status tq_fit_codebook(int bits, float *centroids, float *thresholds);

/* The sphere-coordinate codebook (TQ_VALUE_LAW_SPHERE) of `bits` for vectors
 * of head_dim coordinates (4..1024): the same Lloyd iteration in binary64
 * rounded to binary32, centroids (2^bits) and thresholds (2^bits - 1, may be
 * NULL).  The first fit of a width takes up to ~20 s of host time at 8 bits
 * (head_dim 128 fits are kept for the process). */
tq_status tq_fit_codebook_sphere(int bits, int head_dim, float *centroids, float *thresholds);

/* The value-code lookup table that the one-thread-per-vector compressor uses
 * for a width of 1-4 bits and an ascending threshold set (host; for
 * inspection and tests).  The code of a quotient u is #{j : thresholds[j] < u};
 * the table gives it from u's binary32 bit pattern p:
 *   bits 1-3: entry i = (table[2i], table[2i + 1]) = (t, k) for p >> 22 = i
 *     (sign, exponent, one mantissa bit): k thresholds lie below every u of
 *     the bucket and t is the bit pattern of the bucket's one threshold (+inf
 *     if none): code = k + [t < u];
 *   bits 4: entry i = table[i] = k << 21 | t' for p >> 21 = i (two mantissa
 *     bits): t' the low 21 bits of the bucket's threshold, complemented in
 *     buckets of negative u (2^21 - 1 if none): code = k + [t' < x], x the low
 *     21 bits of p, complemented if u < 0.
 * table: 2048 uint32 (host).  TQ_ERR_ARG for bits outside 1..4 or NULL
 * pointers; TQ_ERR_UNSUPPORTED when a bucket holds two thresholds (the
 * compressor then searches the thresholds instead). */
tq_status tq_value_code_table(int bits, const float *thresholds, uint32_t *table);

/* ------------------------------------------------------------------------ */
/* QJL projection ("TurboMOQ", "QJL residual correction (sub-2-bit)":          */
/* QJLConfig(head_dim, jl_dim); "turboquant-mlx", "RaBitQ vs QJL correction").  */
/* ------------------------------------------------------------------------ */
/* Fill S (host, jl_dim x head_dim floats, row-major) with N(0,1) entries:
 * SplitMix64(seed) words in pairs -> u1 = ((w1>>11)+1) 2^-53, u2 = (w2>>11) 2^-53
 * -> Box-Muller (binary64) -> binary32.  The caller copies S to device memory
 * it owns and passes that copy to tq_compress / tq_decode_attention.
 * jl_dim must be a multiple of 32 and at most 1024 (kernels: jl_dim == 128). */
tq_status tq_make_qjl(int head_dim, int jl_dim, uint64_t seed, float *S);

/* ------------------------------------------------------------------------ */
/* Packed segment layout (one layer, one token range with fixed bit widths).   */
/* ------------------------------------------------------------------------ */
typedef struct {
    int batch;         /* B */
    int n_heads;       /* H (KV heads), 1..TQ_MAX_HEADS */
    int head_dim;      /* d */
    int capacity;      /* tokens the buffers are laid out for */
    int jl_dim;        /* QJL sketch length (bits per key); used if any qjl[h] */
    uint8_t kbits[TQ_MAX_HEADS]; /* per head, 1..8 */
    uint8_t vbits[TQ_MAX_HEADS]; /* per head, 1..8 */
    uint8_t qjl[TQ_MAX_HEADS];   /* per head, 0/1: 1-bit residual sketch of keys */
    uint8_t value_law;           /* value codebook: TQ_VALUE_LAW_GAUSS or TQ_VALUE_LAW_SPHERE
                                  * (the latter fitted for d = 128); anything else is
                                  * TQ_ERR_ARG */
    uint8_t qjl_v[TQ_MAX_HEADS]; /* per head, 0/1: 1-bit sketch of the value residual
                                  * y - sigma c[code] (same S and jl_dim as the keys);
                                  * decode adds sqrt(pi/2)/jl ||r|| S^T s to the value */
} tq_segment_layout;

/* Value codebook laws (the Lloyd-Max quantizer of u = y / RMS(y)):
 *   TQ_VALUE_LAW_GAUSS   N(0,1) ("TurboMOQ", "Architecture": Lloyd-Max codebook)
 *   TQ_VALUE_LAW_SPHERE  sqrt(d) times a coordinate of a uniform unit d-vector,
 *                        density ~ (1 - u^2/d)^((d-3)/2): the exact law of a
 *                        rotated coordinate ("TurboMOQ", "Head-to-Head
 *                        Comparison": Beta-CDF codebook). */
#define TQ_VALUE_LAW_GAUSS 0
#define TQ_VALUE_LAW_SPHERE 1

/* Byte layout (all offsets are multiples of 16 when the bases are aligned):
 *   record sizes rk(h) = d*kbits[h]/8, rv(h) = d*vbits[h]/8 bytes;
 *   kcodes byte offset of (b, h, t) = b*cap*sum_h rk + cap*sum_{h'<h} rk(h')
 *                                     + t*rk(h)      (vcodes likewise with rv);
 *   code i of a vector occupies bits [b*i, b*i+b) of its record (LSB first);
 *   kscale / vscale (float) index (b*H + h)*cap + t  (key: max|y|, value: RMS);
 *   QJL heads ranked q(h) = #{h' < h : qjl[h']}, nq of them: qjl_signs byte
 *   offset ((b*nq + q(h))*cap + t)*jl/8 (bit j LSB-first = sign of (S r)_j >= 0),
 *   qjl_norm (float, ||r||_2) index (b*nq + q(h))*cap + t;
 *   value sketches likewise with v(h) = #{h' < h : qjl_v[h']}, nv of them:
 *   vqjl_signs byte offset ((b*nv + v(h))*cap + t)*jl/8, vqjl_norm index
 *   (b*nv + v(h))*cap + t. */
typedef struct {
    size_t kcode_bytes, vcode_bytes, kscale_bytes, vscale_bytes, qjl_sign_bytes, qjl_norm_bytes;
    size_t vqjl_sign_bytes, vqjl_norm_bytes;
} tq_packed_sizes;

/* Sizes of the device buffers of a packed segment.  TQ_ERR_ARG on an
 * invalid layout (bits outside 1..8, H outside 1..16, capacity < 0, ...). */
tq_status tq_packed_size(const tq_segment_layout *layout, tq_packed_sizes *sizes);

typedef struct {
    void *kcodes, *vcodes;   /* device, sizes from tq_packed_size */
    float *kscale, *vscale;  /* device */
    void *qjl_signs;         /* device, may be NULL when no head uses QJL */
    float *qjl_norm;         /* device, may be NULL when no head uses QJL */
    void *vqjl_signs;        /* device, may be NULL when no head sketches its values */
    float *vqjl_norm;        /* device, may be NULL when no head sketches its values */
} tq_packed_bufs;

/* ------------------------------------------------------------------------ */
/* Compression (rotation -> per-vector scale -> quantize -> pack [-> QJL]).     */
/* ------------------------------------------------------------------------ */
/* K, V: device fp16, element (b, h, t, i) at b*stride_b + h*stride_h +
 * t*stride_t + i (strides in elements; stride_t*2 and every base must be
 * 16-byte aligned).  Compresses n_tokens tokens into positions
 * [t_begin, t_begin + n_tokens) of the packed segment (chunked compression
 * appends with t_begin = tokens already stored).  qjl_S: device jl_dim x
 * head_dim floats from tq_make_qjl, required iff some qjl[h] or qjl_v[h] is set.
 * All arithmetic is IEEE binary32 in a fixed order, so the codes are a pure
 * function of the input:
 *   y = binary32(1/sqrt(d)) * D (butterflies h = 1, 2, ..., d/2 of D x);
 *   keys: m = max|y_i|, r = 1/m (0 if m = 0), code = clamp(floor((y r + 1) 2^(b-1)),
 *         0, 2^b - 1);
 *   values: sigma = sqrt(pairwise-tree sum of y_i^2 / d), r = 1/sigma (0 if 0),
 *         code = #{k : thr_k < y r};
 *   QJL: r_i = y_i - m*((code+1/2) 2^(1-b) - 1), sign bits of S r, ||r||_2;
 *   value QJL: r_i = y_i - sigma*c[code] (binary32 product and difference, c
 *         the binary32 centroids), sign bits of S r, ||r||_2.
 * With a dense rotation (rot->dense) y = Q x runs on the tensor cores: x fp16
 * times Q carried as two fp16 parts (~2^-22), binary32 accumulation in an order
 * the hardware chooses, so a code can differ from the exact product's where y
 * lies within ~1e-6 of a decision boundary; the scales and quantizers are the
 * ones above.  Dense rotation with QJL (key or value) heads, or strides TMA
 * cannot describe, return TQ_ERR_UNSUPPORTED.
 * Returns TQ_ERR_SIZE if t_begin + n_tokens > capacity. */
tq_status tq_compress(const tq_segment_layout *layout, const tq_rotation *rot,
                      const float *qjl_S, const void *K, const void *V, int n_tokens,
                      int64_t stride_b, int64_t stride_h, int64_t stride_t, int t_begin,
                      const tq_packed_bufs *out, void *stream);

/* The dense-rotation compress kernel bounds every wait for its own copies and
 * tensor-core work; one that gave up sets a flag (process-wide, per device).
 * *flag = that flag (waits for the device); reset != 0 clears it.  Returns
 * TQ_ERR_TIMEOUT when the flag was set (before any reset), TQ_OK when not. */
tq_status tq_compress_error_flag(int *flag, int reset);

/* Dequantize token positions [t_begin, t_begin + n_tokens) of a packed segment.
 * k_rot / v_rot (device floats [B][H][n_tokens][d], either may be NULL): the
 * rotated-space values binary32(m * level(code)) and binary32(sigma *
 * centroid[code]).  k_orig / v_orig (may be NULL): the original-space vectors
 * R applied to those (binary32; neither includes a QJL term).  A debugging
 * and parity aid: decode attention never materialises these. */
tq_status tq_dequantize(const tq_segment_layout *layout, const tq_packed_bufs *bufs,
                        const tq_rotation *rot, int t_begin, int n_tokens, float *k_rot,
                        float *v_rot, float *k_orig, float *v_orig, void *stream);

/* Tier demotion ("TurboMOQ", "Progressive temporal tiering": tokens move to
 * tiers with fewer bits as they age).  Tokens [src_t_begin, src_t_begin + n)
 * of a packed segment are dequantized in the rotated space (keys m*level(code),
 * values sigma*centroid[code], binary32) and compressed again with the widths
 * of `dst` into its positions [dst_t_begin, dst_t_begin + n): the same
 * per-vector scales and quantizers as tq_compress, applied to the
 * reconstruction, with no rotation either way.  Both segments must have the
 * same batch, heads and head_dim; dst must carry no QJL heads, key or value
 * (TQ_ERR_UNSUPPORTED; a source's sketches are not carried over); the two segments' buffers must not overlap.  Any
 * widths 1..8 are accepted (demotion normally lowers them).  TQ_ERR_SIZE if a
 * range exceeds its capacity. */
tq_status tq_requantize(const tq_segment_layout *src, const tq_packed_bufs *src_bufs, int src_t_begin,
                        const tq_segment_layout *dst, const tq_packed_bufs *dst_bufs, int dst_t_begin,
                        int n_tokens, void *stream);

/* Progressive tiers by token age ("TurboMOQ", "Progressive temporal tiering"):
 * position p has age n_tokens-1-p; tier i holds ages [bound[i-1], bound[i])
 * (bound[-1] = 0, bound[n_bounds] = infinity).  Writes tier i's position
 * range [start[i], end[i]) for i = 0..n_bounds (empty tiers get start == end). */
tq_status tq_age_tiers(int n_tokens, int n_bounds, const int *age_bounds, int *start,
                       int *end);

/* ------------------------------------------------------------------------ */
/* Decode attention over the compressed cache.                                 */
/* ------------------------------------------------------------------------ */
#define TQ_SEG_PACKED 0
#define TQ_SEG_FP16 1

typedef struct {
    int kind;                  /* TQ_SEG_PACKED or TQ_SEG_FP16 */
    int n_tokens;              /* tokens attended, 0..layout.capacity */
    tq_segment_layout layout;  /* batch/n_heads/head_dim/capacity for both kinds;
                                  bits and qjl for packed segments */
    tq_packed_bufs packed;     /* TQ_SEG_PACKED */
    const void *k16, *v16;     /* TQ_SEG_FP16: fp16 [B][H][capacity][d], unrotated */
    float *attn_mass;          /* optional (NULL: none), device float [B][H][capacity],
                                  16-byte aligned, caller-owned: tq_decode_attention
                                  writes entry (b, h, t), t < n_tokens, with the
                                  attention mass of token t (below) */
} tq_segment;

/* Score estimators for QJL heads (the sketch s = sign(S r), rho = ||r|| is the
 * same for both; q' = R q):
 *   TQ_QJL_UNBIASED   q'.yhat + sqrt(pi/2)/jl * rho * <S q', s>  ("TurboMOQ",
 *                     "QJL residual correction (sub-2-bit)"; unbiased)
 *   TQ_QJL_SIGN_PAIR  q'.yhat + (pi/2)/jl * ||q'|| * rho * <sign(S q'), s>
 *                     ("turboquant-mlx", "RaBitQ vs QJL correction": pi/2 times
 *                     both scales times the sign agreement; sign(0) = +1).  Its
 *                     mean is ||q'|| rho (pi/2 - theta), theta the angle of q'
 *                     and r (Sheppard): unbiased only to first order in cos theta. */
#define TQ_QJL_UNBIASED 0
#define TQ_QJL_SIGN_PAIR 1

typedef struct {
    tq_rotation rot;           /* the layer's rotation (same D for K, V and q) */
    int n_segments;            /* 0..TQ_MAX_SEGMENTS; order does not matter */
    tq_segment seg[TQ_MAX_SEGMENTS];
    int qjl_estimator;         /* TQ_QJL_UNBIASED or TQ_QJL_SIGN_PAIR (else TQ_ERR_ARG) */
} tq_layer_view;

/* Bytes of device workspace tq_decode_attention needs for these layers. */
tq_status tq_decode_workspace_size(const tq_layer_view *layers, int n_layers, int batch,
                                   int n_heads, int q_heads, int head_dim, size_t *bytes);

/* out[l][b][j][:] = softmax_t(q_j . k_t / sqrt(d)) . v_t over every token of
 * every segment of layer l, where query head j reads KV head j/(q_heads/n_heads)
 * and, for packed tokens, k_t = R (yhat_k [+ rhat_QJL]) and v_t = R yhat_v.
 * Computed without materialising k_t, v_t: q is rotated once, scores and the
 * value sum run in the rotated space on the packed codes (split over token
 * chunks with an online softmax), and one inverse rotation is applied to the
 * merged value sum.  QJL heads add the layer's qjl_estimator term to q'.yhat.
 * q: device fp16 [n_layers][batch][q_heads][d]; out: device float, same shape.
 * qjl_S: device jl_dim x d floats, required iff a packed segment uses QJL.
 * workspace: device, >= tq_decode_workspace_size bytes (TQ_ERR_SIZE otherwise).
 * The call copies a small plan (host -> workspace) with cudaMemcpyAsync from
 * one of the library's pinned staging buffers (so the host does not wait for
 * the stream), then launches its kernels on `stream`: the QJL query prep (if
 * any QJL segment), the fp16-segment split-K kernel (if any fp16 segment) and
 * one persistent split-K kernel per (key bits, value bits, QJL) class of the
 * packed segments, each merging the partials of the (layer, batch, KV head)
 * it completes.  A layer with no tokens yields zeros.
 * Attention mass (the per-token signal of attention-weighted tier demotion,
 * "TurboMOQ", "Attention-weighted tier demotion"): for every segment with
 * attn_mass set, one more kernel after the merges writes
 *   attn_mass[b][h][t] = (1/g) sum_{j : j/g = h} p_j(t),
 * p_j(t) the softmax weight of token t for query head j (g = q_heads/n_heads),
 * so that over all segments of a layer sum_t attn_mass[b][h][t] = 1; scores are
 * recomputed from the codes in binary32 and normalised by the merged max and
 * sum. */
tq_status tq_decode_attention(const tq_layer_view *layers, int n_layers, int batch,
                              int n_heads, int q_heads, int head_dim, const float *qjl_S,
                              int jl_dim, const void *q, float *out, void *workspace,
                              size_t ws_bytes, void *stream);

/* The kernels never spin without bound: a split-K CTA that waits too long for
 * its own shared-memory copies (never expected) stops, lets the copies it
 * issued land, leaves its part of the output unwritten (no merge completes for
 * the (layer, batch, KV head) groups it touched) and sets a flag at the start
 * of the workspace.  This call synchronises `stream` and stores that flag
 * (0 = no such event) in *flag; it returns TQ_ERR_TIMEOUT when the flag is set
 * and TQ_OK when not.  workspace = NULL reads the flag of this device's static
 * scratch array (the one tq_decode_attention_static uses).  The next decode
 * call on the same workspace clears it. */
tq_status tq_decode_error_flag(const void *workspace, int *flag, void *stream);

/* Failure-path hook, for tests of the timeout handling: the number of polls a
 * split-K CTA makes while waiting for a stage of its own copies before it gives
 * up (default and maximum 2^20; 0 makes every such wait give up at once, while
 * the drain of the copies already issued keeps the full bound, so that no copy
 * outlives its CTA).  Applies to later tq_decode_attention calls of the
 * process.  TQ_ERR_ARG outside [0, 2^20]. */
tq_status tq_set_decode_wait_polls(int polls);

/* Measurement hook: when both events are non-NULL, every later
 * tq_decode_attention call on this host thread records `start` on its stream
 * just before the split-K kernel over packed segments and `stop` just after it,
 * so the caller can time that kernel alone with cudaEventElapsedTime.  Pass
 * NULL, NULL to turn it off.  The events are cudaEvent_t handles owned by the
 * caller; no effect on results. */
tq_status tq_set_decode_kernel_events(void *start, void *stop);

/* Kernel launches the calling thread's last decode call made (query prep,
 * split-K grids, attention mass), for callers that account for them. */
int tq_decode_last_launches(void);

/* ------------------------------------------------------------------------ */
/* Decode attention without a caller-supplied workspace.  (No counterpart on   */
/* the pages: this entry point exists for callers, not for the method.)        */
/* ------------------------------------------------------------------------ */
/* Bytes of the library's own scratch array.  A device commits it when the
 * array's module is loaded there -- with the CUDA runtime's default lazy
 * loading, at the first tq_decode_attention_static call (or static flag read)
 * on that device -- and holds it until the process exits. */
#define TQ_STATIC_WORKSPACE_BYTES (16u << 20)

/* Same result and same kernels as tq_decode_attention, for callers that may not
 * allocate device memory while they run: serving loops that reserve all their
 * device memory at start-up and forbid cudaMalloc afterwards (it can synchronize
 * the device and fragment a budgeted pool), or hosts whose device memory is
 * owned by another framework's allocator.  The scratch (plan, rotated queries,
 * split-K partials) is a fixed array of TQ_STATIC_WORKSPACE_BYTES inside the
 * library instead of a caller buffer; the caller still passes q and out.  The
 * call allocates no device memory (its plan upload uses the library's pinned
 * host staging buffers, allocated by the first decode calls of the process).
 *   - Set-up: the first call on a device, with that device current, loads the
 *     array (committing its TQ_STATIC_WORKSPACE_BYTES of device memory), looks up
 *     its device address (cudaGetSymbolAddress) and caches it.  Make that first
 *     call (a warm-up on a small cache) during start-up, before reserving the
 *     rest of the device memory for a pool and before any stream capture.
 *   - Limit: returns TQ_ERR_SIZE, before launching anything, when the call needs
 *     more scratch than TQ_STATIC_WORKSPACE_BYTES (tq_decode_workspace_size tells
 *     how much); split the layers over several calls or use tq_decode_attention.
 *     Argument and alignment errors come first, as for tq_decode_attention.
 *   - Timeouts: tq_decode_error_flag(NULL, ...) reads the array's flag.
 *   - Sharing: every call uses the same array, which keeps the previous call's
 *     contents; nothing in it needs to start at zero (each call writes all it
 *     reads).  Calls that overlap on the GPU -- on different streams or from
 *     different host threads -- race on the array: order them on one stream.
 * Other arguments and errors as for tq_decode_attention. */
tq_status tq_decode_attention_static(const tq_layer_view *layers, int n_layers, int batch,
                                     int n_heads, int q_heads, int head_dim, const float *qjl_S,
                                     int jl_dim, const void *q, float *out, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* TQ_H */
