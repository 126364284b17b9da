/*
 * qmv.h - C ABI of the GB300 quantized small-batch matvec / MoE library.
 *
 * The operation: LLM decode multiplies a handful of token activations
 * (1 to 64 rows) by block-quantized weight matrices that are consumed in
 * their compressed form, dequantized on the fly.  The pages this library is
 * built from name the pieces:
 *   - small-batch matvecs for K-quants, IQ4_XS and Q8_0 (with a split-K
 *     variant) for 1..16 tokens: "Castagna Veloce", section "Kernels for the
 *     MI50", third bullet;
 *   - i-quant MoE decode kernels for batches up to 64 tokens and the
 *     expert-grouped quantized MoE scheme: same section, first two bullets;
 *   - gate/up + SwiGLU fusion and Q8 activations reused across weight types:
 *     "Castagna Veloce", section "Fused operations", fourth and fifth bullets;
 *   - a decode row is a matrix-vector product bound by weight reads, and the
 *     hot path must consume compressed weights directly: "Running GLM-5.3 on
 *     Two 8-GPU AMD W7900D Machines", sections "A single decode row is not a
 *     large matrix multiplication" and "Keep quantized weights compressed in
 *     memory";
 *   - effective bandwidth = weight bytes / kernel time: same page, section
 *     "A faster kernel can still leave the full chain slower" (the paragraph
 *     under the constraint table).
 * The pages give no byte layouts; the layouts below are this library's own.
 *
 * ------------------------------------------------------------------------
 * Conventions shared by every entry point
 * ------------------------------------------------------------------------
 *   - Activations X are fp32 row-major [n_tok][K]; outputs Y are fp32
 *     row-major [n_tok][M]:  Y[t][m] = sum_k What[m][k] * Xhat[t][k].
 *   - A weight matrix W has M rows; row m occupies qmv_row_bytes(fmt, K)
 *     contiguous bytes starting at W + m * qmv_row_bytes(fmt, K).  A row of
 *     a quantized format is a sequence of GROUPS; every group is a 16-byte
 *     header followed by its payload, so every group (and row) starts on a
 *     16-byte boundary.  (F16 / F32 rows are plain arrays of K values.)
 *   - Every pointer argument is device memory owned by the caller (unless a
 *     comment says otherwise).  The library allocates nothing, keeps no
 *     per-call state and never synchronises the stream (except
 *     qmv_get_device_error).  Calls are stream-ordered and asynchronous.
 *   - Calls may come from several host threads at once (the library's
 *     per-device lookups are made once under a lock; the only shared device
 *     buffer is qmv_splitk_run_static's scratch array, see there).
 *   - Every data pointer must be 16-byte aligned (QMV_ERR_ALIGN otherwise).
 *   - Return value: 0 on success, a negative QMV_ERR_* code on a host-side
 *     argument error (nothing is launched then).  Errors detected on the
 *     device (bad expert ids, a stalled pipeline) set a device error word,
 *     read with qmv_get_device_error(); kernels never trap.
 *
 * ------------------------------------------------------------------------
 * Activation quantization (shared by every weight format)
 * ------------------------------------------------------------------------
 *   Per token, per 32-element block j of x (K % 32 == 0):
 *     amax = max_i |x_i|                         (exact)
 *     d    = amax / 127                          (fp32, IEEE round-to-nearest)
 *     id   = (d > 0) ? 1 / d : 0                 (fp32, IEEE round-to-nearest)
 *     q_i  = clamp(rne(x_i * id), -127, 127)     (fp32 product, then round
 *                                                 half to even to an integer)
 *     s    = sum_i q_i                           (int32)
 *   and Xhat_i = d * q_i.  (A block whose amax is below about 3.7e-37 has a
 *   subnormal d whose reciprocal overflows to infinity: its nonzero elements
 *   get +-127 and its zero elements, 0 * inf being no number, get 0.)
 *   Non-finite x is outside the contract.
 *
 * ------------------------------------------------------------------------
 * Weight formats (values are What; fp16 fields are IEEE binary16, little
 * endian; bit strings are little endian across bytes)
 * ------------------------------------------------------------------------
 * QMV_Q8_0: blocks of 32 weights, What = d * q, d fp16, q int8.
 *   Group = 8 blocks (256 weights), 272 bytes:
 *     header  bytes [2j, 2j+2)        : d of block j (j = 0..7)
 *     payload bytes [16j, 16j+16)     : q_0..q_15 of block j (int8)
 *             bytes [128+16j, 144+16j): q_16..q_31 of block j
 *   K % 256 == 0; row bytes = 272 * K / 256.
 *
 * QMV_Q4_K: superblocks of 256 weights = 8 sub-blocks of 32,
 *   What = d * sc_j * q - dmin * m_j, q in [0,15], sc_j, m_j in [0,63].
 *   Group = 1 superblock, 144 bytes:
 *     header  bytes 0-1 : d (fp16);  bytes 2-3: dmin (fp16)
 *             bytes 4-15: 96-bit string; bits [12j, 12j+6) = sc_j and
 *                         bits [12j+6, 12j+12) = m_j  (j = 0..7)
 *     payload bytes [16j, 16j+16): sub-block j; byte i holds q_i in its low
 *                         nibble and q_{i+16} in its high nibble (i = 0..15)
 *   K % 256 == 0; row bytes = 144 * K / 256.
 *
 * QMV_IQ4_XS: superblocks of 256 weights = 8 sub-blocks of 32,
 *   What = d * (ls_j - 32) * CB[c], c in [0,15], ls_j in [0,63], with the
 *   int8 codebook CB = {-127,-104,-83,-65,-49,-35,-22,-10,
 *                       1,13,25,38,53,69,89,113}.
 *   Group = 2 superblocks (512 weights), 272 bytes:
 *     header  bytes [8s, 8s+2)  : d of superblock s (s = 0,1)
 *             bytes [8s+2, 8s+8): 48-bit string, bits [6j, 6j+6) = ls_j
 *     payload bytes [128s + 16j, +16): superblock s, sub-block j, nibbles
 *                         arranged as for QMV_Q4_K (byte i: c_i | c_{i+16}<<4)
 *   K % 512 == 0; row bytes = 272 * K / 512.
 *
 * QMV_Q5_K ("Castagna Veloce", section "Kernels for the MI50": small-batch
 *   matvecs for the K-quants q4_K, q5_K, q6_K): superblocks of 256 weights
 *   = 8 sub-blocks of 32, What = d * sc_j * q - dmin * m_j, q in [0,31],
 *   sc_j, m_j in [0,63].  Group = 1 superblock, 176 bytes:
 *     header  bytes 0-15 : as QMV_Q4_K (d, dmin, the sc / m string)
 *     high    bytes [16+4j, 20+4j): sub-block j, a 32-bit little-endian
 *                         word whose bit i is bit 4 of q_i
 *     payload bytes [48+16j, 64+16j): sub-block j; byte i holds bits 0-3 of
 *                         q_i in its low nibble and of q_{i+16} in its high
 *   K % 256 == 0; row bytes = 176 * K / 256.  Dense matvecs only (not an
 *   expert format of moe_qmv_run).
 *
 * QMV_Q6_K (same passage): superblocks of 256 weights = 16 sub-blocks of
 *   16, What = d * sc_i * (q - 32), q in [0,63], sc_i in [0,127].  Each code
 *   is stored as v = (q - 32) mod 64 (6-bit two's complement).
 *   Group = 1 superblock, 208 bytes:
 *     header  bytes 0-1 : d (fp16);  bytes 2-15: 112-bit string, bits
 *                         [7i, 7i+7) = sc_i (i = 0..15)
 *     high    bytes [16+8j, 24+8j): 32-weight block j (sub-blocks 2j, 2j+1),
 *                         two 32-bit little-endian words, the first for
 *                         weights 0..15, the second for 16..31; weight e of a
 *                         word (k = e / 4, b = e % 4) has bits 4-5 of its v at
 *                         bits [8b + 2k, 8b + 2k + 2)
 *     payload bytes [80+16j, 96+16j): block j; byte i holds bits 0-3 of v_i
 *                         in its low nibble and of v_{i+16} in its high
 *   K % 256 == 0; row bytes = 208 * K / 256.  Dense matvecs only.
 *
 * QMV_Q8_G64, QMV_Q8_G128 ("Running GLM-5.3 on Two 8-GPU AMD W7900D
 *   Machines", section "Why 4-bit today: room for 5/6-bit, but not FP8": KV in
 *   Q8G64, the LM head in Q8G128): What = d_s * q, q int8, one fp16 d_s
 *   per 64 (G64) or 128 (G128) consecutive weights.  Group = 8 scale groups
 *   (512 or 1024 weights), 16 + 512 = 528 or 16 + 1024 = 1040 bytes:
 *     header  bytes [2s, 2s+2): d_s (s = 0..7)
 *     payload bytes [256h, 256h+256) after the header: weights 256h..256h+255
 *             of the group, laid out as a QMV_Q8_0 payload (block j of the
 *             256: q_0..15 at 16j, q_16..31 at 128+16j)
 *   K % 512 (G64) or K % 1024 (G128) == 0.  Dense matvecs only.
 *
 * QMV_F16, QMV_F32 ("Castagna Veloce", section "Kernels for the MI50": the
 *   small-batch matvec also serves F16 and F32 weights): unquantized rows,
 *   What = w, IEEE binary16 or binary32, weight k at bytes [2k, 2k+2) or
 *   [4k, 4k+4) of the row.  There is no header and no activation
 *   quantization: these formats take x as it is (Xhat = x, fp32), every
 *   product and sum in fp32 (same accuracy bound).  K % 32 == 0; row bytes
 *   = 2 K or 4 K.  Dense matvecs only (qmv_run, qmv_splitk_run[_static],
 *   qmv_run_residual, qmv_run_siblings; not qmv_run_q8, not the MoE pool).
 *   Their activations are staged in shared memory as fp32 for a CTA's whole
 *   K-range, so long rows take fewer tokens per pass (more passes over the
 *   weights), and qmv_run takes rows of up to about 24K weights; split-K
 *   shortens the range (qmv_splitk_choose picks enough splits for the
 *   fp32 activations of one pass of up to 16 tokens to take at most 96 KB).
 *
 * Bytes per weight: Q8_0 1.0625, Q4_K 0.5625, IQ4_XS 0.53125, Q5_K 0.6875
 * (the same densities as the GGML formats of the same names), Q6_K 0.8125
 * (7-bit sub-scales instead of GGML's 8-bit ones), Q8_G64 1.03125, Q8_G128
 * 1.015625, F16 2, F32 4; GGUF byte compatibility is not a goal.
 */
#ifndef QMV_H
#define QMV_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

enum qmv_format {
  QMV_Q8_0 = 0,
  QMV_Q4_K = 1,
  QMV_IQ4_XS = 2,
  QMV_Q5_K = 3,
  QMV_Q6_K = 4,
  QMV_Q8_G64 = 5,
  QMV_Q8_G128 = 6,
  QMV_F16 = 7,
  QMV_F32 = 8
};

enum qmv_status {
  QMV_OK = 0,
  QMV_ERR_FORMAT = -1,    /* unknown format code */
  QMV_ERR_SHAPE = -2,     /* M <= 0, K not a multiple of the group size, ... */
  QMV_ERR_NTOK = -3,      /* n_tok not in [1, 64] or top_k not in [1, 8] */
  QMV_ERR_NULL = -4,      /* a required pointer is NULL */
  QMV_ERR_ALIGN = -5,     /* a pointer is not 16-byte aligned */
  QMV_ERR_WORKSPACE = -6, /* workspace too small */
  QMV_ERR_CUDA = -7,      /* a CUDA runtime call or launch failed */
  QMV_ERR_DEVICE = -8,    /* no usable sm_103 device */
  QMV_ERR_UNAVAILABLE = -9 /* the call needs a build this library was not made as */
};

/* Device error word bits (qmv_get_device_error). */
#define QMV_DEVERR_EXPERT_RANGE 0x1 /* an expert id outside [0, n_experts) */
#define QMV_DEVERR_EXPERT_DUP 0x2   /* an expert id repeated within a token */
#define QMV_DEVERR_TIMEOUT 0x4      /* a pipeline wait exceeded its limit */
#define QMV_DEVERR_RANGE 0x8        /* debug build: an access failed its range check (and was skipped) */

#define QMV_MAX_TOKENS 64
#define QMV_MAX_PREFILL_TOKENS 16384 /* moe_qmv_prefill_run */
#define QMV_MAX_TOPK 8

/* Bytes of one quantized row of K weights; negative QMV_ERR_* if fmt or K is
 * invalid. */
int64_t qmv_row_bytes(int fmt, int64_t K);

/* Quantize fp32 weights w [M][K] (device) into format fmt, writing
 * M * qmv_row_bytes(fmt, K) bytes at W (device).  Per block the scale is
 * chosen from the block's range and each code is the nearest grid point
 * (ties to the even / lower code), all in fp64:
 *   Q8_0  : d = fp16(amax / 127); q = rne(w / d) clamped to [-127,127].
 *   Q4_K  : per sub-block lo = min(0, min w), hi = max w, a = (hi-lo)/15,
 *           b = -lo; d = fp16(max a / 63), dmin = fp16(max b / 63);
 *           sc = rne(a / d), m = rne(b / dmin) clamped to [0,63];
 *           q = argmin_{0..15} |w - (d*sc*q - dmin*m)| (ties: lower q).
 *   IQ4_XS: per sub-block s = amax / 113; d = fp16(max s / 31);
 *           ls = 32 + clamp(rne(s / d), 0, 31);
 *           c = argmin_{0..15} |w - d*(ls-32)*CB[c]| (ties: lower c).
 *   F16   : fp16(w) per weight;  F32: w as it is.
 * (fp16(.) rounds to nearest even; a zero scale gives zero codes.)  This is a
 * preparation step, not part of the decode hot path. */
int qmv_quantize_weights(int fmt, const float* w, int64_t M, int64_t K, void* W,
                         cudaStream_t stream);

/* Activation quantization (rule above) of x [n_tok][K] into the library's
 * Q8 activation layout: q int8 [n_tok][K], d fp32 [n_tok][K/32] and sum
 * int32 [n_tok][K/32], where d and sum are per block in order and the codes
 * of each 256-element group (8 blocks) are stored halves first: element p of
 * block l of the group at byte (p / 16) * 128 + l * 16 + p % 16 of the
 * group.  (That is the order the matvec kernels read, so qmv_run_q8 brings
 * the rows into shared memory with bulk copies.)  K % 256 == 0,
 * 1 <= n_tok <= 64.  "Q8 activations reused across weight types": the
 * result feeds qmv_run_q8 for any weight format. */
int qmv_quantize_act(const float* x, int64_t K, int n_tok, int8_t* q, float* d,
                     int32_t* sum, cudaStream_t stream);

/* Y[t][m] = sum_k What[m][k] * Xhat[t][k] for t < n_tok, m < M: the
 * small-batch quantized matvec.  x fp32 [n_tok][K] is quantized inside the
 * kernel (rule above); every integer block dot product is exact and the block
 * scales are applied in fp32 (F16 / F32 weights: Xhat = x, fp32 products).
 * Accuracy: |Y - Y_exact| <= 1e-5 * sum_k |What[m][k] * Xhat[t][k]|.
 * 1 <= n_tok <= 64.  Tokens run in passes of up to 16; for QMV_Q4_K a pass
 * of 5 to 16 tokens forms its integer block dot products on the tensor
 * cores (f16 operands holding the integers, fp32 accumulation: exact) and
 * applies the scales by the same fp32 formula, in a different summation
 * order than passes of 1 to 4 tokens. */
int qmv_run(int fmt, const void* W, const float* x, float* y, int64_t M,
            int64_t K, int n_tok, cudaStream_t stream);

/* Same as qmv_run with pre-quantized activations (the layout of
 * qmv_quantize_act); results are bitwise equal to qmv_run on the x they
 * were quantized from.  Quantized formats only (QMV_F16 / QMV_F32:
 * QMV_ERR_FORMAT). */
int qmv_run_q8(int fmt, const void* W, const int8_t* xq, const float* xd,
               const int32_t* xs, float* y, int64_t M, int64_t K, int n_tok,
               cudaStream_t stream);

/* Split-K matvec for few-row, long-K shapes: K is cut into n_split contiguous
 * ranges of whole groups; pass 1 writes partial sums partial[s][t][m] into
 * the workspace, pass 2 adds them in the fixed order s = 0..n_split-1, so the
 * result is bitwise reproducible for a given (shape, n_tok, n_split).
 * n_split = 0 picks a split count from the shape (qmv_splitk_choose).
 * ws must hold qmv_splitk_workspace_bytes(M, n_tok, n_split) bytes (none
 * for n_split = 1).  If it holds that (rounded up to 256) plus
 * qmv_act_q8_bytes(K, n_tok) more and the call has more than 8 tokens, or
 * 5-8 tokens with a split, K > 4096 or M >= 7168 (the shapes where it
 * measured faster), the activations are quantized once into the rest of the
 * workspace (one more kernel launch) and each CTA copies its K-range in
 * instead of quantizing it again: the same arithmetic (bitwise equal
 * results), less work per CTA. */
size_t qmv_act_q8_bytes(int64_t K, int n_tok);
int qmv_splitk_choose(int fmt, int64_t M, int64_t K, int n_tok);
size_t qmv_splitk_workspace_bytes(int64_t M, int n_tok, int n_split);
int qmv_splitk_run(int fmt, const void* W, const float* x, float* y, int64_t M,
                   int64_t K, int n_tok, int n_split, void* ws, size_t ws_bytes,
                   cudaStream_t stream);

/* Matvec plus residual ("Castagna Veloce", section "Fused operations":
 * matvec + residual add): y[t][m] = (What Xhat)[t][m] + r[t][m], the fp32
 * addition made once, after the dot product is complete (in the matvec's
 * store, or in the ordered second pass of split-K).  r fp32 [n_tok][M]
 * (device, 16-byte aligned) may be y itself (y += What Xhat).  Arguments,
 * workspace and split choice as qmv_splitk_run; r NULL -> QMV_ERR_NULL. */
int qmv_run_residual(int fmt, const void* W, const float* x, const float* r, float* y,
                     int64_t M, int64_t K, int n_tok, int n_split, void* ws,
                     size_t ws_bytes, cudaStream_t stream);

/* Sibling matvecs sharing one x ("Castagna Veloce", section "Fused
 * operations": batched sibling matvecs, and Q8 activations reused across
 * weight types): y_i = What_i Xhat for i < count, each W_i of format fmts[i]
 * with M[i] rows of the same K weights (K a multiple of every format's group
 * size), x fp32 [n_tok][K], y_i fp32 [n_tok][M[i]].  fmts, W, M and y are
 * host arrays of count (1..QMV_MAX_SIBLINGS) entries; the matrices and
 * outputs are device memory.  From 4 tokens the activations are quantized
 * once into ws (at least qmv_act_q8_bytes(K, n_tok) bytes, 16-byte aligned)
 * and every matvec copies them in; with fewer tokens each matvec quantizes
 * them while staging and ws may be NULL.  One launch per matvec (plus the
 * quantizer), chained by programmatic dependent launch.  Results are
 * bitwise those of qmv_run on each W_i. */
#define QMV_MAX_SIBLINGS 8
int qmv_run_siblings(int count, const int* fmts, const void* const* W, const int64_t* M,
                     float* const* y, const float* x, int64_t K, int n_tok, void* ws,
                     size_t ws_bytes, cudaStream_t stream);

/* qmv_splitk_run for callers that cannot allocate device memory (the pages
 * have no counterpart to this entry point; it exists for embedding).  Some
 * callers may not call cudaMalloc: a plugin running while its host framework
 * captures a CUDA graph (allocation is not allowed during capture), or a host
 * that owns all device memory.  This variant takes no workspace: the partial
 * sums go to a static device array of QMV_STATIC_SCRATCH_BYTES that the
 * library holds on every GPU that loads it, until the process exits.  With a
 * split above one and more than 4 tokens, the activations quantized once
 * (qmv_act_q8_bytes(K, n_tok)) are placed in the array too, after the
 * partial sums, when both fit (as qmv_splitk_run does with a large enough
 * workspace).
 *   - Rejects split shapes whose partial sums exceed that size with
 *     QMV_ERR_WORKSPACE (qmv_splitk_workspace_bytes(M, n_tok, n_split) must
 *     be <= QMV_STATIC_SCRATCH_BYTES; n_split = 0 picks the split as
 *     qmv_splitk_run does, n_split = 1 uses no scratch).
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture.
 *   - Every call shares the array: calls that can overlap on the GPU (other
 *     streams, concurrently launched graphs) race, on the partial sums and
 *     the quantized activations alike.  Nothing needs clearing: each call
 *     overwrites every value it reads.
 *   - Allocates nothing (no cudaMalloc / cudaFree, no allocating library).
 * Results are bitwise equal to qmv_splitk_run with the same n_split. */
#define QMV_STATIC_SCRATCH_BYTES (8u << 20)
int qmv_splitk_run_static(int fmt, const void* W, const float* x, float* y,
                          int64_t M, int64_t K, int n_tok, int n_split,
                          cudaStream_t stream);

/* Expert pool of one MoE FFN layer. */
typedef struct moe_experts {
  int32_t n_experts;   /* E */
  int32_t hidden;      /* H: K of gate/up, M of down */
  int32_t ffn;         /* F: rows of gate (and of up), K of down */
  int32_t fmt_gate_up; /* QMV_Q8_0, QMV_Q4_K or QMV_IQ4_XS */
  int32_t fmt_down;    /* QMV_Q8_0, QMV_Q4_K or QMV_IQ4_XS */
  int32_t reserved;
  const void* w_gate_up; /* [E][2F rows][row_bytes(fmt_gate_up, H)]:
                            rows 0..F-1 gate, rows F..2F-1 up */
  const void* w_down;    /* [E][H rows][row_bytes(fmt_down, F)] */
} moe_experts;

/* Expert-grouped MoE decode layer:
 *   for each token t and slot k < top_k with expert e = ids[t][k]:
 *     g = Wgate_e Xhat_t,  u = Wup_e Xhat_t          (F values each)
 *     h = silu(g) * u,  silu(z) = z / (1 + exp(-z))  (fp32)
 *     o_{t,k} = Wdown_e Hhat_{t,k}                   (Hhat: h quantized by
 *                                                     the activation rule)
 *   y[t] = sum_{k=0..top_k-1} gates[t][k] * o_{t,k}, added in k order.
 * ids int32 [n_tok][top_k], gates fp32 [n_tok][top_k], x fp32 [n_tok][H],
 * y fp32 [n_tok][H].  The slots routed to one expert are computed in groups
 * of up to G slots, G a power of two up to 16 chosen from the mean load
 * n_tok * top_k / n_experts (at least 8 from 4 tokens on); each group streams
 * the expert's weights once, so an expert with more than G slots in the call
 * is streamed once per group (ceil(slots / G) times); the groups of one
 * expert run side by side, so the repeats are served from L2 (measured on
 * GB300 with 64 tokens on the same 8 experts, 8 groups each: 1.02x / 1.11x
 * one read per expert from DRAM for gate/up / down).  A slot whose id is outside
 * [0, n_experts) or repeats an earlier id of the same token contributes 0 and
 * sets the device error word.  gates are used as given (not renormalised).
 * The workspace holds the intermediates at the offsets of
 * moe_qmv_workspace_offsets (slot p = t * top_k + k; rows of slots that do
 * not route are left unwritten):
 *   [0] h  f32 [n_tok*top_k][F]     (SwiGLU output)
 *   [1] hq int8 [n_tok*top_k][F]    (h quantized by the activation rule)
 *   [2] hd f32 [n_tok*top_k][F/32]  [3] hs i32 [n_tok*top_k][F/32]
 *   [4] o  f32 [n_tok*top_k][H]     (down projection of each slot)
 * Constraints: H and F multiples of the group sizes of the two formats,
 * n_experts <= 512, 1 <= n_tok <= 64, 1 <= top_k <= 8, top_k <= n_experts. */
size_t moe_qmv_workspace_bytes(const moe_experts* e, int n_tok, int top_k);
int moe_qmv_workspace_offsets(const moe_experts* e, int n_tok, int top_k,
                              size_t offsets[5]);
int moe_qmv_run(const moe_experts* e, const int32_t* ids, const float* gates,
                const float* x, float* y, int n_tok, int top_k, void* ws,
                size_t ws_bytes, cudaStream_t stream);

/* The same MoE layer for large batches (prefill, "Castagna Veloce", section
 * "Kernels for the MI50", second bullet: the expert-grouped quantized MoE
 * GEMM for prompt processing), 1 <= n_tok <= QMV_MAX_PREFILL_TOKENS, on the
 * tcgen05 tensor cores: per routed expert, tiles of 128 weight rows times up
 * to 64 of its token slots; each 32-weight block's integer dot products are
 * formed exactly by the tensor core (the codes of weights and activations
 * held as f16, accumulated in fp32) and its fp32 scales applied as in
 * moe_qmv_run, so the result satisfies the same bounds (h within the gate/up
 * tolerance, q8(h) by the activation rule, o and y within 1e-5 *
 * sum |What Hhat| times the gates).  Arguments and the meaning of ids, gates,
 * x and y as moe_qmv_run; each expert's weights are read once per 64 of its
 * slots.  The workspace holds h, its quantization and o at the offsets
 * moe_qmv_prefill_workspace_offsets returns (the five entries of
 * moe_qmv_workspace_offsets), plus the quantized x and the per-expert slot
 * lists.  Constraints as moe_qmv_run, and hidden and ffn multiples of 128.
 * Five launches, no programmatic dependent launch. */
size_t moe_qmv_prefill_workspace_bytes(const moe_experts* e, int n_tok, int top_k);
int moe_qmv_prefill_workspace_offsets(const moe_experts* e, int n_tok, int top_k, size_t offsets[5]);
int moe_qmv_prefill_run(const moe_experts* e, const int32_t* ids, const float* gates, const float* x, float* y,
                        int n_tok, int top_k, void* ws, size_t ws_bytes, cudaStream_t stream);

/* Router and top-k ("Castagna Veloce", section "Fused operations": router
 * and top-k in one kernel, i.e. matvec, gating, top-k and weight
 * normalization), producing the ids and gates moe_qmv_run takes:
 *   logits[t][e] = What_r[e] . Xhat[t]   (the quantized matvec of qmv_run:
 *                                        n_experts rows of `hidden` weights
 *                                        in format fmt, x fp32 [n_tok][hidden])
 *   ids[t][0..top_k): the top_k experts of token t in decreasing order of
 *     logit; of equal logits the lower expert index comes first;
 *   gates[t][k], normalised over the picked experts:
 *     QMV_GATING_SOFTMAX: exp(l_k - l_0) / sum_j exp(l_j - l_0)
 *     QMV_GATING_SIGMOID: s_k / sum_j s_j,  s = 1 / (1 + exp(-l)).
 * logits fp32 [n_tok][n_experts] is written too (caller-owned device memory):
 * the picks are decided on exactly these values.  ids int32 and gates fp32
 * [n_tok][top_k].  Two launches (the matvec, then one warp per token for
 * gating, top-k and normalisation), chained by programmatic dependent launch.
 * Constraints: hidden a multiple of the format's group size, 1 <= top_k <= 8,
 * top_k <= n_experts <= 512, 1 <= n_tok <= 64, gating one of the two values
 * (else QMV_ERR_SHAPE); all pointers 16-byte aligned device memory. */
#define QMV_GATING_SOFTMAX 0
#define QMV_GATING_SIGMOID 1
int moe_route_run(int fmt, const void* Wr, const float* x, int n_experts, int64_t hidden,
                  int n_tok, int top_k, int gating, float* logits, int32_t* ids, float* gates,
                  cudaStream_t stream);

/* Diagnostic (no counterpart on the pages): the activation quantizer uses
 * branch-free FMA sequences for d = amax / 127 and 1 / d; this compares them
 * with the IEEE round-to-nearest division and reciprocal on every
 * non-negative float of their ranges and ADDS the mismatch counts to
 * mismatches[0] (division) and mismatches[1] (reciprocal), device memory,
 * 16-byte aligned.  Both must stay 0. */
int qmv_check_rounding(unsigned long long* mismatches, cudaStream_t stream);

/* Diagnostic (no counterpart on the pages): Df = A B^T for one 128 x N
 * tile of int8 codes over one 32-element block, through the tcgen05 tensor
 * cores with the codes held exactly as f16 and an fp32 accumulator (the
 * tcgen05 MMA of sm_103a has no int8 kind).  A int8 [128][32], B int8
 * [N][32], Df fp32 [128][N], row-major device memory; 16 <= N <= 256,
 * N % 16 == 0.  Every product and partial sum is an integer below 2^24 in
 * magnitude, so Df equals the exact integer dot products. */
int qmv_tc_probe(const int8_t* A, const int8_t* B, int N, float* Df, cudaStream_t stream);

/* Diagnostic: measured issue rates per SM per SM clock (median over the
 * SMs, one CTA per SM, clock64 around a fixed amount of work):
 *   [0] dp4a, [1] prmt, [2] fp32 FMA, [3] packed fp32x2 FMA, [4] int32 to
 *   fp32 conversion (thread instructions per clock);
 *   [5] mma.sync m16n8k32 s8, [6] mma.sync m16n8k16 f16 (multiply-adds);
 *   [7], [8], [9] tcgen05 f16 MMA, M = 128, N = 256, 64, 32 (multiply-adds).
 * Writes min(count, 10) values to the host array rates and returns how many
 * (or a negative QMV_ERR_*).  scratch: device memory of at least
 * qmv_measure_pipes_scratch_bytes() bytes, 16-byte aligned.  Synchronises
 * the stream. */
size_t qmv_measure_pipes_scratch_bytes(void);
int qmv_measure_pipes(double* rates, int count, void* scratch, size_t scratch_bytes, cudaStream_t stream);

/* Diagnostic (no counterpart on the pages): the library's bounded wait, made
 * to run out.  Every mbarrier wait in the kernels gives up after about 2^31
 * SM cycles (about a second), sets QMV_DEVERR_TIMEOUT and returns, so a
 * stalled pipeline never hangs the GPU; the limit is a compile-time constant
 * of the kernels, whose hot loops then carry no other code.  This launches
 * one warp that runs the same wait loop, with limit_cycles (1 .. 2^31) as its
 * limit, on an mbarrier that nothing ever completes: it gives up, sets
 * QMV_DEVERR_TIMEOUT in the device error word and returns.  cycles (device,
 * may be NULL) receives the SM cycles the wait lasted (at least
 * limit_cycles).  The context stays usable. */
int qmv_wait_probe(long long limit_cycles, unsigned long long* cycles, cudaStream_t stream);

/* Debug builds (the library compiled with QMV_DEBUG, e.g. by the package's
 * build(debug=True)) check every global access of the kernels against the
 * extent of its buffer, which the host derives from the call's arguments
 * (y: n_tok x M, the split partials, the workspace parts, ...), and every
 * shared-memory access against the CTA's allocation; an access that fails
 * its check is skipped and sets QMV_DEVERR_RANGE.  This stands in for a
 * memory checker: no check traps.  This call makes every later call hand the
 * extents of its result buffers (y, logits, ids, gates, the quantizers'
 * outputs; not the workspace) to those checks n elements short (n = 0
 * restores them), so that in-bounds stores near the end fail their checks:
 * a test of the checks that touches no memory out of bounds (the stores into
 * the results' last n elements are then skipped).  Release builds:
 * QMV_ERR_UNAVAILABLE.  Not thread-safe with respect to calls in flight. */
int qmv_debug_shrink_outputs(int64_t n);

/* Synchronises `stream`, then reads and clears the device error word
 * (QMV_DEVERR_* bits, 0 if none) into *err. */
int qmv_get_device_error(cudaStream_t stream, int* err);

/* Static description of a status code. */
const char* qmv_strerror(int code);

#ifdef __cplusplus
}
#endif
#endif /* QMV_H */
