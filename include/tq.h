/*
 * tq.h - C ABI of libtq: TurboQuant / PolarQuant KV-cache compression and
 * attention computed directly over the compressed cache, for NVIDIA GB300
 * (sm_103a).
 *
 * The method (per key or value vector x of length d, in blocks of `block`
 * coordinates; block == d gives one norm per vector, block == 32 gives the
 * "block-32" layout):
 *   1. split off the norm n = ||x_j|| of every block and quantise u = x_j/n
 *      ("TurboQuant From Scratch on Real KV Tensors", section 2, step 1);
 *   2. rotate y = H D u with D a random +-1 diagonal and H the orthonormal
 *      Walsh-Hadamard matrix (same section, step 2; ``fwht`` listing);
 *   3. scalar-quantise every y_i with the Lloyd-Max codebook of N(0, 1/block)
 *      (same section, step 3);
 *   4. optionally keep the 1-bit QJL residual sign(S r), r = u - Q(u), plus
 *      ||r|| ("turboquant-pytorch" README, QJL estimator formula);
 *   5. bit-pack the codes with one fp16 scale per block (llama.cpp-turboquant
 *      docs/turboquant.md, "How it works" and "GGML Types": 14-byte turbo3
 *      and 18-byte turbo4 blocks of 32 values).
 *
 * Conventions for every call below:
 *   - Every call returns 0 (TQ_OK) or a negative tq_status; none throws,
 *     none synchronises the device, none allocates memory.  Device work is
 *     enqueued on `stream` (a cudaStream_t passed as void*; NULL = the
 *     legacy default stream).  Errors are reported for invalid arguments
 *     before anything is enqueued; TQ_ERR_CUDA reports a failed launch
 *     (cudaGetLastError right after it).
 *   - The caller owns every buffer.  "device" pointers must be CUDA device
 *     (or managed) memory, 16-byte aligned unless stated otherwise; "host"
 *     pointers are ordinary host memory.
 *   - fp16 values travel as uint16_t bit patterns (IEEE binary16).
 *   - Reserved fields must be zero.
 */
#ifndef TQ_H_
#define TQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TQ_OK = 0,
  TQ_ERR_ARG = -1,          /* NULL pointer, bad shape or stride           */
  TQ_ERR_UNSUPPORTED = -2,  /* (head_dim, block, bits, qjl_m) not handled  */
  TQ_ERR_ALIGN = -3,        /* pointer not aligned as required             */
  TQ_ERR_WORKSPACE = -4,    /* workspace missing or too small              */
  TQ_ERR_CUDA = -5,         /* kernel launch failed                        */
  TQ_ERR_TIMEOUT = -6       /* a bounded device-side wait gave up          */
} tq_status;

typedef enum { TQ_F16 = 0, TQ_F32 = 1 } tq_dtype;

typedef enum { TQ_CODEBOOK_GAUSSIAN = 0, TQ_CODEBOOK_BETA = 1 } tq_codebook_kind_t;

/* Codec settings of one cache (K or V).
 *   head_dim      d in {64, 128, 256}
 *   block         rotation + norm block: a power of two >= 32 dividing d
 *                 (d: one norm per vector; 32: block-32)
 *   bits          MSE bits per coordinate, 1..4, or 8 (one byte per code:
 *                 the 256-level Gaussian codebook, no QJL; the keys of
 *                 "TurboQuant From Scratch"'s k8v4 setting, Finding 1 and
 *                 Takeaways)
 *   qjl_m         0 = no QJL residual; else m rows of S, a multiple of 32,
 *                 <= 256, and block must equal head_dim
 *   norm_correct  0/1: store n / ||reconstructed direction|| instead of n,
 *                 so that the decoded block has the input's norm
 *                 ("TurboQuant From Scratch", section 2, "Norm correction")
 *   codebook      TQ_CODEBOOK_GAUSSIAN (0): Lloyd-Max for N(0, 1/block);
 *                 TQ_CODEBOOK_BETA (1): Lloyd-Max for the exact law of one
 *                 coordinate of a random unit vector in R^block, i.e.
 *                 (x + 1)/2 ~ Beta((block-1)/2, (block-1)/2)
 *                 (llama.cpp-turboquant, "How it works"); other values are
 *                 TQ_ERR_ARG
 *   sign_seed     seed of D: the i-th splitmix64 output (state = seed)
 *                 gives D_i = -1 when its top bit is set, else +1.  Block j
 *                 uses D[j*block .. (j+1)*block). */
typedef struct {
  int32_t head_dim;
  int32_t block;
  int32_t bits;
  int32_t qjl_m;
  int32_t norm_correct;
  int32_t codebook;
  uint64_t sign_seed;
} tq_layout;

/* Packed record of one vector (all little endian):
 *   codes:   d*bits/8 bytes = d/32 groups of 32 rotated coordinates, in
 *            coordinate order; group = `bits` 32-bit words; word w, nibble k
 *            (bits 4k..4k+3) holds
 *              bits=4: code(8w+k)
 *              bits=3: bits 0-2 = code(8w+k), bit 3 = bit w of code(24+k)
 *              bits=2: bits 0-1 = code(8w+k), bits 2-3 = code(16+8w+k)
 *              bits=1: bit p = code(8p+k)
 *            and bits=8: byte i of the record = code(i).
 *            where code(i) = #{k : y_i > beta_k} indexes the ascending
 *            centroids of the Lloyd-Max codebook.
 *   scales:  d/block fp16 values (n, or the norm-corrected value).
 *   qjl:     qjl_m/8 bytes = m/32 words, bit i of word w = [(S r)_{32w+i} >= 0].
 *   rnorm:   one fp16 ||r|| (QJL only).
 * Bytes per element with block 32: 0.4375 at 3 bits, 0.5625 at 4 bits. */

/* Lloyd-Max codebook of N(0, 1/block) with 2^bits levels, solved in double
 * precision on the host and rounded to nearest float (bits 1..8; 16 levels
 * or fewer by the Lloyd iteration, more by Newton's method on the same
 * fixed point).  centroids: host,
 * 2^bits floats, ascending; boundaries: host, 2^bits - 1 midpoints.
 * "TurboQuant From Scratch", section 2, step 3; section 3 (distortion
 * about 0.118 / 0.0345 / 0.0095 at 2 / 3 / 4 bits). */
int tq_codebook(int bits, int block, float* centroids, float* boundaries);

/* The codebook of a layout's `codebook` kind in double precision (host):
 * TQ_CODEBOOK_GAUSSIAN is tq_codebook_f64; TQ_CODEBOOK_BETA solves
 * Lloyd-Max for the density (1 - x^2)^((block-3)/2) / B(1/2, (block-1)/2)
 * on [-1, 1] (block a power of two in 32..256, else TQ_ERR_UNSUPPORTED).
 * boundaries may be NULL. */
int tq_codebook_kind(int bits, int block, int kind, double* centroids, double* boundaries);

/* Same codebook without the rounding to float (host, double). */
int tq_codebook_f64(int bits, int block, double* centroids, double* boundaries);

/* Sign vector D of a layout: out[i] = +1 or -1 for i < d (host int8). */
int tq_signs(uint64_t sign_seed, int d, int8_t* out);

/* Per-vector sizes of a layout (host outputs, any may be NULL): bytes of
 * packed codes, number of fp16 scales, bytes of QJL sign bits. */
int tq_layout_sizes(const tq_layout* layout, int64_t* code_bytes_per_vec,
                    int64_t* scales_per_vec, int64_t* qjl_bytes_per_vec);

/* Quantise n_vec vectors (device).
 *   x            device, row i at x + i*x_row_stride elements, x_dtype
 *                fp16 or fp32; rows of d contiguous elements; the row
 *                start must be 16-byte aligned.
 *   S            device fp32 [qjl_m, d] row major (QJL only, else NULL)
 *   codes        device [n_vec, code_bytes_per_vec]
 *   scales       device fp16 [n_vec, d/block]
 *   qjl_bits     device [n_vec, qjl_m/8]   (QJL only, else NULL)
 *   qjl_rnorm    device fp16 [n_vec]       (QJL only, else NULL)
 * Steps: norm split, y = H D u, code = #{k : y > beta_k}, optional norm
 * correction and QJL, pack (llama.cpp-turboquant, "How it works", Encode).
 * A zero block gets scale 0 (and, with QJL, rho 0 and all sign bits 1). */
int tq_quantize_kv(const tq_layout* layout, const void* x, tq_dtype x_dtype, int64_t n_vec,
                   int64_t x_row_stride, const float* S, uint8_t* codes, uint16_t* scales,
                   uint8_t* qjl_bits, uint16_t* qjl_rnorm, void* stream);

/* Quantise new tokens straight into their slots of a preallocated cache
 * (device).  Every key and value is quantised as it enters the cache
 * ("TurboQuant From Scratch on Real KV Tensors", section 1, the cache
 * update); this is tq_quantize_kv with the output records placed by
 * position instead of by input order.
 *   x            device, B*H*n_new rows ordered (b, h, j), row i at
 *                x + i*x_row_stride elements, x_dtype fp16 or fp32, 16-byte
 *                aligned rows (as tq_quantize_kv)
 *   pos          device int32 [B]: token j of (b, h) goes to cache slot
 *                pos[b] + j; slots outside [0, S_cap) are not written
 *                (nothing else is touched)
 *   page_table, page_size, pages_per_seq
 *                NULL, 0, 0 for a contiguous [B, H, S_cap] cache, else the
 *                paging of tq_kv_view (slot t of batch b is row t % page_size
 *                of page page_table[b*pages_per_seq + t/page_size]; S_cap
 *                <= pages_per_seq*page_size)
 *   codes, scales, qjl_bits, qjl_rnorm
 *                the cache arrays in the tq_kv_view layout
 *   S            device fp32 [qjl_m, d] (QJL only, else NULL)
 * Returns TQ_ERR_ARG for negative sizes or a NULL pos, the tq_quantize_kv
 * errors otherwise; B*H*n_new == 0 is a no-op.  The records written are
 * identical to tq_quantize_kv of the same rows. */
int tq_append_kv(const tq_layout* layout, const void* x, tq_dtype x_dtype, int B, int H, int n_new,
                 int64_t x_row_stride, const int32_t* pos, int64_t S_cap, const int32_t* page_table,
                 int page_size, int pages_per_seq, const float* S, uint8_t* codes, uint16_t* scales,
                 uint8_t* qjl_bits, uint16_t* qjl_rnorm, void* stream);

/* Decode n_vec packed vectors (device) into out [n_vec, d] (fp16 or fp32):
 * x~ = scale * D H (c + [QJL] rho sqrt(pi/2)/m H D S^T (2s - 1)), i.e.
 * unpack -> centroid lookup -> inverse rotation -> x scale
 * (llama.cpp-turboquant, "How it works", Decode; "TurboQuant From
 * Scratch", section 2, un-rotation and QJL term). */
int tq_dequantize_kv(const tq_layout* layout, const uint8_t* codes, const uint16_t* scales,
                     const uint8_t* qjl_bits, const uint16_t* qjl_rnorm, const float* S,
                     int64_t n_vec, void* out, tq_dtype out_dtype, void* stream);

/* A packed cache, all pointers device.
 *   page_table == NULL: [B, Hkv, S_cap] vectors, tokens contiguous within a
 *     (batch, head): record (b, h, t) is vector index (b*Hkv + h)*S_cap + t
 *     of the per-vector arrays above.
 *   page_table != NULL (paged): the arrays hold pages of page_size tokens,
 *     [num_pages, Hkv, page_size] vectors; token t of batch b lives in page
 *     p = page_table[b*pages_per_seq + t/page_size] (device int32) at record
 *     (p*Hkv + h)*page_size + t % page_size.  page_size is a positive
 *     multiple of 32, S_cap must be <= pages_per_seq*page_size, and the K and
 *     V views of one call share page_table, page_size and pages_per_seq
 *     (else TQ_ERR_ARG).  Pages of a sequence need not be contiguous or
 *     ordered; entries of the table past a sequence's length are not read. */
typedef struct {
  const uint8_t* codes;
  const uint16_t* scales;
  const uint8_t* qjl_bits;   /* NULL unless layout.qjl_m > 0 */
  const uint16_t* qjl_rnorm; /* NULL unless layout.qjl_m > 0 */
  const float* S;            /* NULL unless layout.qjl_m > 0 */
  tq_layout layout;
  const int32_t* page_table; /* NULL: contiguous [B, Hkv, S_cap] */
  int32_t page_size;
  int32_t pages_per_seq;
} tq_kv_view;

/* Fused decode attention over the packed cache: one query per
 * (batch, q-head), q fp16 [B, Hq, d] device, out fp16 [B, Hq, d] device.
 * q-head h reads KV head h / (Hq/Hkv); batch b attends positions
 * [0, kv_len[b]) (kv_len: device int32 [B], or NULL for ctx everywhere;
 * every kv_len[b] must be <= ctx <= S_cap).  softmax_scale <= 0 selects
 * 1/sqrt(d).  Scores are formed in the rotated domain, <H D q, c> scaled
 * by the block norms, V is accumulated rotated and rotated back once per
 * output ("llama.cpp-turboquant", "Fused tile path": K side <Hc,q> =
 * <c,Hq>, V side sum p_j H c_j = H sum p_j c_j); online fp32 softmax with
 * the context split into n_split parts merged by log-sum-exp
 * (n_split = 0: chosen by the library).  workspace: device, at least
 * tq_decode_workspace_bytes(...) bytes, 16-byte aligned.  With QJL keys the
 * score adds ||k|| rho sqrt(pi/2)/m <S q, 2s - 1> ("turboquant-pytorch",
 * QJL estimator formula).  8-bit keys are read by the CUDA-core kernel;
 * 8-bit values, and QJL values beside 8-bit keys, are TQ_ERR_UNSUPPORTED. */
int tq_decode_attn(const tq_kv_view* K, const tq_kv_view* V, const uint16_t* q, int B, int Hq,
                   int Hkv, int64_t S_cap, const int32_t* kv_len, int64_t ctx,
                   float softmax_scale, uint16_t* out, void* workspace, size_t workspace_bytes,
                   int n_split, void* stream);

/* Size of the library-owned scratch array used by tq_decode_attn_static. */
#define TQ_DECODE_STATIC_SCRATCH_BYTES (8u << 20)

/* tq_decode_attn for callers that cannot allocate device memory.  No
 * counterpart in the source pages: it exists for callers whose device
 * memory is owned by someone else (a serving runtime or plugin host that
 * hands out all memory from its own pool and forbids cudaMalloc after
 * start-up) or who cannot pay for the implicit synchronisation of an
 * allocation on their hot path.  Same arguments and results as
 * tq_decode_attn without workspace / workspace_bytes: the split-K partials
 * go to a file-scope device array of TQ_DECODE_STATIC_SCRATCH_BYTES bytes
 * inside libtq, which every GPU that loads the library keeps until the
 * process exits.  Nothing is allocated, neither here nor by the caller.
 *   - Sizes whose partials need more than that (tq_decode_workspace_bytes)
 *     are refused with TQ_ERR_WORKSPACE before anything is enqueued.
 *   - The first call on a device looks up that device's copy of the array
 *     (cudaGetSymbolAddress, with the device current) and caches it; make
 *     that first call before any stream capture.  A failed lookup returns
 *     TQ_ERR_CUDA and clears the runtime's last error, so later calls do
 *     not see it.  cudaDeviceReset on that device invalidates the cached
 *     address: do not call this function on the device after a reset.
 *   - All calls on a device share the one array and it keeps the last
 *     call's contents (no call needs it zeroed): calls that overlap on the
 *     GPU (other streams, other host threads) race on it and must be
 *     serialised by the caller. */
int tq_decode_attn_static(const tq_kv_view* K, const tq_kv_view* V, const uint16_t* q, int B, int Hq,
                          int Hkv, int64_t S_cap, const int32_t* kv_len, int64_t ctx,
                          float softmax_scale, uint16_t* out, int n_split, void* stream);

/* Workspace bytes for tq_decode_attn with these sizes (host).  n_split = 0
 * gives the size for the library's own choice; *n_split_out (may be NULL)
 * receives the largest split count that choice takes for these sizes (the
 * count used depends on the layouts: each kernel splits the context to fill
 * one wave of its own CTAs, so a call may use fewer). */
int tq_decode_workspace_bytes(int B, int Hq, int Hkv, int head_dim, int64_t ctx, int n_split,
                              size_t* bytes, int* n_split_out);

/* Decode attention over the packed cache plus an unquantised fp16 residual
 * window of the most recent tokens ("TurboQuant From Scratch on Real KV
 * Tensors", Finding 5: the last tokens kept in full precision).  Batch b
 * attends, in one softmax, to the cache tokens [0, min(ctx, kv_len[b])) and
 * the window tokens [0, win_len[b]) (win_len NULL: win for every batch);
 * attention does not depend on the order of the tokens.
 *   k_win, v_win  device fp16 [B, Hkv, W_cap, head_dim]: unquantised keys and
 *                 values in the original (unrotated) domain, 8-byte aligned;
 *                 caller-owned, read only
 *   W_cap         window slots per (batch, KV head), >= 0
 *   win_len       device int32 [B] or NULL; entries are clamped to [0, W_cap]
 *   win           window tokens of every batch when win_len is NULL,
 *                 0 <= win <= W_cap
 * The other arguments are tq_decode_attn's.  workspace: at least
 * tq_decode_window_workspace_bytes(...) bytes, 16-byte aligned.  The window's
 * softmax partial is one split slot more, rotated into V's coded domain and
 * merged by the same combine.  Errors: TQ_ERR_ARG for a missing window
 * array, W_cap < 0 or win outside [0, W_cap]; TQ_ERR_ALIGN for window
 * arrays that are not 8-byte aligned; otherwise as tq_decode_attn. */
int tq_decode_attn_window(const tq_kv_view* K, const tq_kv_view* V, const uint16_t* q, int B, int Hq,
                          int Hkv, int64_t S_cap, const int32_t* kv_len, int64_t ctx,
                          const uint16_t* k_win, const uint16_t* v_win, int W_cap,
                          const int32_t* win_len, int win, float softmax_scale, uint16_t* out,
                          void* workspace, size_t workspace_bytes, int n_split, void* stream);

/* GGML-style blocks (llama.cpp-turboquant, "GGML Types" and "How it
 * works"): the packed cache of a layout without QJL rewritten as blocks of
 * 32 values, each the fp16 norm of the values' rotation block (little-endian)
 * followed by their packed codes (the group's 4*bits bytes of this library's
 * layout): 2 + 4*bits bytes, 14 at 3 bits and 18 at 4 bits.  With a 128-value
 * rotation block (and the Beta codebook of a 128-value chunk, codebook 1)
 * this is the page's turbo3/turbo4 arrangement: the chunk's norm is in each
 * of its four blocks.  tq_from_blocks takes a rotation block's norm from its
 * first 32-value block.
 *   codes   device [n_vec, head_dim*bits/8], 4-byte aligned
 *   scales  device fp16 [n_vec, head_dim/block], 2-byte aligned
 *   blocks  device [n_vec, head_dim/32, 2 + 4*bits] bytes, 2-byte aligned
 * TQ_ERR_UNSUPPORTED for QJL layouts. */
int tq_to_blocks(const tq_layout* layout, const uint8_t* codes, const uint16_t* scales, int64_t n_vec,
                 uint8_t* blocks, void* stream);
int tq_from_blocks(const tq_layout* layout, const uint8_t* blocks, int64_t n_vec, uint8_t* codes,
                   uint16_t* scales, void* stream);

/* Decode attention read straight from caches in the block form above, with
 * no conversion of the cache ("llama.cpp-turboquant", "Token generation
 * degrades with context depth" and "Fused tile path": a bulk conversion
 * costs O(context) per generated token; decoding the blocks inside the
 * attention kernel avoids it).  Same arguments, results and workspace
 * (tq_decode_workspace_bytes) as tq_decode_attn, with each cache given as
 * its layout and its blocks:
 *   k_blocks, v_blocks  device [B, Hkv, S_cap, head_dim/32, 2 + 4*bits]
 *                       bytes (tq_to_blocks of a contiguous cache),
 *                       2-byte aligned, else TQ_ERR_ALIGN
 *   q, out, workspace   16-byte aligned, as for tq_decode_attn
 * Runs the CUDA-core split kernel for every group size 1, 2, 4, 8.  Layouts
 * with QJL or 8-bit codes, and other group sizes, are TQ_ERR_UNSUPPORTED. */
int tq_decode_attn_blocks(const tq_layout* k_layout, const uint8_t* k_blocks, const tq_layout* v_layout,
                          const uint8_t* v_blocks, const uint16_t* q, int B, int Hq, int Hkv, int64_t S_cap,
                          const int32_t* kv_len, int64_t ctx, float softmax_scale, uint16_t* out,
                          void* workspace, size_t workspace_bytes, int n_split, void* stream);

/* Recursive polar-angle quantizer ("TurboQuant: 3-Bit Compression with Zero
 * Overhead", Part 1: the recursive polar transformation and its quantisation
 * step), a codec of its own beside the rotation + Lloyd-Max one.  A vector
 * of head_dim = 2^k values becomes its L2 norm and head_dim - 1 angles:
 * level 1 pairs coordinates (x[2i], x[2i+1]) into radius sqrt(x0^2 + x1^2)
 * and angle atan2(x1, x0), every further level pairs the previous radii the
 * same way.  Each angle is stored as the index k of the nearest point
 * k / (2^b - 1) * 2 pi - pi of a uniform grid over [-pi, pi] (ties to even).
 *   x        device rows of x_row_stride elements (fp16 or fp32, 2/4-byte
 *            aligned); row i holds vector i
 *   codes    device [n_vec, head_dim*bits/8] bytes, 16-byte aligned: the
 *            angle indices level by level (level 1 first, the root's last,
 *            then one 0 index), packed like the MSE codes (32-code groups of
 *            nibble words, see tq_kv_view)
 *   radius   device fp16 [n_vec], 2-byte aligned
 * head_dim 64, 128 or 256 and bits 1-4, else TQ_ERR_UNSUPPORTED.
 * Dequantisation rebuilds the tree from the root: a radius r with angle t
 * gives the children r cos(t), r sin(t); out is [n_vec, head_dim] fp16 or
 * fp32, 16-byte aligned. */
int tq_polar_code_bytes(int head_dim, int bits, int64_t* code_bytes);
int tq_polar_quantize(const void* x, int x_dtype, int64_t n_vec, int head_dim, int64_t x_row_stride, int bits,
                      uint8_t* codes, uint16_t* radius, void* stream);
int tq_polar_dequantize(const uint8_t* codes, const uint16_t* radius, int64_t n_vec, int head_dim, int bits,
                        void* out, int out_dtype, void* stream);

/* Workspace bytes for tq_decode_attn_window with these sizes (host). */
int tq_decode_window_workspace_bytes(int B, int Hq, int Hkv, int head_dim, int64_t ctx, int n_split,
                                     size_t* bytes);

/* Prefill attention: Tq queries per (batch, q-head) at positions
 * ctx-Tq .. ctx-1 over cache positions [0, ctx); q fp16 [B, Hq, Tq, d],
 * out fp16 [B, Hq, Tq, d], both device.  causal != 0: query i attends
 * positions <= ctx-Tq+i (bottom-right aligned).  K/V tiles are decoded into
 * shared memory (rotated domain, scaled) and QK^T / PV run on the tensor
 * cores ("llama.cpp-turboquant", "Prompt processing": the conversion
 * amortises over the query batch).  QJL and 8-bit codes are not supported
 * here (TQ_ERR_UNSUPPORTED).  workspace: device, >= tq_prefill_workspace_bytes. */
int tq_prefill_attn(const tq_kv_view* K, const tq_kv_view* V, const uint16_t* q, int B, int Hq,
                    int Hkv, int Tq, int64_t S_cap, int64_t ctx, int causal, float softmax_scale,
                    uint16_t* out, void* workspace, size_t workspace_bytes, void* stream);

int tq_prefill_workspace_bytes(int B, int Hq, int Hkv, int head_dim, int Tq, int64_t ctx,
                               size_t* bytes);

/* ---- Device-side waits and status ----------------------------------------
 * The tensor-core prefill (tq_prefill_attn) and the fast quantiser
 * (tq_quantize_kv / tq_append_kv with fp16 input, block 32 or 64, 2-4 bits,
 * no QJL) hand work between the warps of a CTA through mbarriers, and every
 * such wait is bounded.  A wait longer than the wait limit records
 * TQ_ERR_TIMEOUT in the library's device status word for that device and
 * goes on waiting, so the launch still completes and its outputs are valid;
 * a call returns before its kernels run, so this is the only way a caller
 * learns of it.  A wait longer than the hard bound (2 s, or the limit if
 * larger) stops its CTA: the fast quantiser first waits for every load and
 * product it has in flight, then stops with its outputs incomplete; the
 * prefill stops without that drain (a device that has stopped making
 * progress).  Either way the status word says TQ_ERR_TIMEOUT. */

/* Sets the wait limit, in nanoseconds, for launches issued after the call
 * (process-wide, all devices); 0 restores the default of 2 s.  Always
 * returns TQ_OK. */
int tq_set_wait_limit_ns(uint64_t ns);

/* Reads the device status word of `device`: *status = TQ_OK when no launch
 * of this library recorded a failure since the last clear, else the first
 * failure recorded (TQ_ERR_TIMEOUT).  It first synchronises the device, so
 * every launch issued before the call is counted; clear != 0 resets the word
 * after reading.  The calling thread's current device is left unchanged.
 * Returns TQ_ERR_ARG for a NULL status or an invalid device, TQ_ERR_CUDA
 * when the synchronisation or the read fails (a fault of an earlier launch
 * shows up here). */
int tq_device_status(int device, int clear, int* status);

/* Human-readable text of a tq_status (static storage). */
const char* tq_strerror(int status);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int tq_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TQ_H_ */
