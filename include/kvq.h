/*
 * kvq.h -- C ABI of the low-bit KV-cache library (libkvq.so).
 *
 * One operation family: single-token decode attention over a key/value cache
 * whose older tokens are stored as asymmetric uniform INT4, INT3 or INT2 codes and
 * whose most recent Nr tokens stay fp16 (and, optionally, whose first tokens
 * stay fp16 as an attention-sink window).
 *
 * Sources the operations follow (web pages on low-bit KV-cache decoding):
 *   - "Tensor Core accelerated low-bit KV cache decoding" (BitDecoding page),
 *     section 2.1: scale = (max - min) / (2^b - 1), code = round((K - min) / scale).
 *   - same page, section 2.2: residual partition, K_pack = KV[:L-Nr] quantized,
 *     K_res = KV[L-Nr:] kept fp16.
 *   - same page, section 2.3: GQA query regrouping, one KV read serves gq query heads.
 *   - same page, section 3.1: per-thread min/max, warp shuffle reduction, pack in registers.
 *   - same page, section 5.1: cache pointers aligned to 128 bytes.
 *   - "KV cache quantization InnerQ" page, section 2.1: groups of G = 32 along the
 *     inner (head_dim) dimension, one row shares its group parameters.
 *   - same page, section 2.2: hybrid mode, each group quantized symmetrically or
 *     asymmetrically, whichever reconstructs it better, with a 1-bit mode mask.
 *   - same page, section 2.3: recent-token window; a new token enters the window and,
 *     when the window is full, its oldest token is quantized into the main cache.
 *     Also the attention-sink window: the first tokens stay in full precision, set
 *     at prefill and fixed afterwards.
 *   - same page, section 3.1: dequantized value = scale * q + zero.
 *   - same page, section 3.2: 32 consecutive head_dim values packed together.
 *   - TurboQuant 3-bit article, section 3.1: eight 3-bit codes in 24 bits; section
 *     6.1: a paged cache of 32-token blocks.
 *
 * ---------------------------------------------------------------------------
 * Notation
 *   B   batch (sequences)             Hkv  KV heads        Hq  query heads (Hq % Hkv == 0)
 *   gq  = Hq / Hkv                    d    head_dim (multiple of 32, 32..256)
 *   G   = 32 group size along d       Ng   = d / 32 groups per token and head
 *   b   bits per code, 2, 3 or 4      Nr   fp16 residual window length (0..1024)
 *   cap packed-token capacity per (sequence, KV head)
 *   S   fp16 attention-sink window length (0..256)
 *   P   page size of a paged cache (0: contiguous, 32: paged), NP pages in its pool
 *
 * ---------------------------------------------------------------------------
 * Memory layout (all arrays are plain device memory owned by the caller; K and V
 * each have their own four arrays with identical shapes)
 *
 *   codes    uint8  [B][Hkv][cap][d*b/8]
 *            One token row holds d codes as a little-endian bit string: element
 *            e (0 <= e < d) occupies bits [e*b, e*b + b) of the row, so group g
 *            is the contiguous bytes [g*4*b, (g+1)*4*b): 16 bytes for INT4, 12 for
 *            INT3, 8 for INT2.
 *            INT4 byte k = c[2k] | c[2k+1] << 4.
 *            INT3: eight codes per 3 bytes, a code may straddle two bytes.
 *            INT2 byte k = c[4k] | c[4k+1] << 2 | c[4k+2] << 4 | c[4k+3] << 6.
 *            Paged caches (P = 32): codes, params and mode bytes live in a pool of
 *            NP pages, codes uint8 [NP][Hkv][32][d*b/8] (params, mode likewise); packed
 *            token t of sequence b, KV head h is row t % 32 of head h in page
 *            block_table[b][t / 32].  cap must be a multiple of 32.
 *   params   uint32 [B][Hkv][cap][Ng]
 *            One half2 per group: low 16 bits = scale (fp16), high 16 bits =
 *            min (fp16).  Dequantized value x^ = min + code * scale.
 *   residual fp16   [B][Hkv][Nr][d]
 *            Ring of the most recent tokens, kept in full precision.
 *   sink     fp16   [B][Hkv][S][d]
 *            The first sink_len[b] tokens of sequence b, kept in full precision.
 *   mode     uint8  [B][Hkv][cap]   (hybrid caches only)
 *            Bit g of a packed row's byte = mode of its group g: 1 asymmetric,
 *            0 symmetric.  Both modes dequantize as min + code * scale, so
 *            decode does not read it.
 *   block_table int32 [B][cap / 32]   (paged caches only): page of each 32 packed tokens.
 *   packed_len, res_len, res_head, sink_len   int32 [B]   (device)
 *            Per sequence: packed tokens, residual tokens, ring slot of the oldest
 *            residual token, sink tokens.  Sequence b attends over
 *            sink_len[b] + packed_len[b] + res_len[b] tokens.
 *   err_word uint32 (device, sticky bit set, see KVQ_ERRBIT_*)
 *
 * Every device pointer must be 16-byte aligned (KVQ_ERR_MISALIGNED otherwise);
 * 128-byte alignment is recommended.
 *
 * ---------------------------------------------------------------------------
 * Quantization rule, per (sequence, head, token, group) with fp16 inputs x_0..x_31
 *   Q1  mn = min_j x_j, mx = max_j x_j
 *   Q2  scale_f = ((float)mx - (float)mn) / (float)(2^b - 1)   fp32, round-to-nearest-even divide
 *   Q3  scale_h = fp16_rne(scale_f) (subnormals kept); min_h = fp16(mn + 0.0f) (-0 stored as +0)
 *   Q4  s = (float)scale_h; code_j = 0 if s == 0, else
 *       clamp(rint(((float)x_j - (float)mn) / s), 0, 2^b - 1)   fp32 subtract and divide,
 *       rint = round half to even
 *   Q5  pack as in the layout above
 * Hybrid caches (desc.hybrid = 1) replace Q1-Q4 per group by H1-H3:
 *   H1  symmetric candidate: a = max_j |x_j|, h = 2^(b-1), scale_s = fp16_rne(a / (h - 1))
 *       (fp32 divide), s = (float)scale_s, t_j = clamp(rint(x_j / s), -(h-1), h-1)
 *       (fp32 divide; 0 if s == 0), code = t_j + h, min_s = fp16(-h * s + 0.0f).
 *   H2  error of a candidate (fp32, each operation rounded, no fused multiply-add):
 *       e_j = x_j - (min + (float)code_j * scale); S_q = sum of e_j^2 over
 *       j = 8q .. 8q+7 in index order; E = (S_0 + S_1) + (S_2 + S_3).
 *   H3  the symmetric candidate is stored when min_s is finite and E_s < E_a; otherwise
 *       the asymmetric one (Q1-Q4).  Mode bit 0 = symmetric, 1 = asymmetric.
 *   Q6  with ns = min(S, L) and nr = min(Nr, L - ns): tokens [0, ns) are copied to the
 *       sink, tokens [ns, L - nr) are packed into slots [0, L - ns - nr), the last nr
 *       are copied to the residual ring in order, res_head = 0.
 *
 * Decode: O[b][hq] = softmax(q[b][hq] . K^T / sqrt(d)) V over the sink tokens, the
 * dequantized packed tokens and the residual tokens of KV head hq / gq, returned as fp16.
 *
 * ---------------------------------------------------------------------------
 * Conventions
 *   Ownership: the caller owns all memory and the stream.  The library allocates
 *     nothing and never synchronizes, except kvq_read_error.
 *   Streams: `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *   Errors: argument errors return synchronously and launch nothing.  A failed
 *     launch returns KVQ_ERR_CUDA.  Data-dependent errors (capacity overflow, an
 *     empty sequence, a bounded wait that ran out) set bits in *err_word on the
 *     device; kvq_read_error reads and clears them.
 */
#ifndef KVQ_H_
#define KVQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KVQ_OK = 0,
  KVQ_ERR_INVALID_ARG = 1, /* a bad shape, a NULL pointer, a size mismatch */
  KVQ_ERR_UNSUPPORTED = 2, /* a valid but unsupported configuration (bits, d, gq) */
  KVQ_ERR_MISALIGNED = 3,  /* a device pointer that is not 16-byte aligned */
  KVQ_ERR_CAPACITY = 4,    /* a sequence does not fit in the packed capacity */
  KVQ_ERR_CUDA = 5,        /* a CUDA runtime call or launch failed */
  KVQ_ERR_TIMEOUT = 6,     /* a bounded device-side wait ran out */
  KVQ_ERR_EMPTY = 7        /* decode over a sequence with no tokens */
} kvq_status;

/* Bits of *err_word (sticky until kvq_read_error clears them). */
#define KVQ_ERRBIT_CAPACITY 0x1u /* pack or append would pass cap; the token was dropped */
#define KVQ_ERRBIT_EMPTY 0x2u    /* decode saw a sequence with no tokens; output zeroed */
#define KVQ_ERRBIT_TIMEOUT 0x4u  /* a bounded wait gave up; that CTA wrote nothing */
#define KVQ_ERRBIT_BADLEN 0x8u   /* seq_lens[b] < 0 or > Lmax; that sequence was skipped */
#define KVQ_ERRBIT_BADPAGE 0x10u /* a block-table page outside [0, NP): pack/append wrote nothing
                                   there; decode output of that sequence is undefined */

/* Static description of one layer's cache.  group must be 32.  Every field is
 * significant: zero-initialise the struct (sink = 0 keeps no sink window). */
typedef struct {
  int32_t batch;        /* B   >= 1 */
  int32_t num_kv_heads; /* Hkv >= 1 */
  int32_t head_dim;     /* d: multiple of 32, 32..256 */
  int32_t bits;         /* b: 2, 3 or 4 */
  int32_t group;        /* G: 32 */
  int32_t capacity;     /* packed tokens per (sequence, KV head), >= 0 */
  int32_t residual;     /* Nr: 0..1024 */
  int32_t sink;         /* S: 0..256, first tokens kept fp16 (attention-sink window) */
  int32_t hybrid;       /* 0: asymmetric groups; 1: hybrid sym/asym groups with a mode mask */
  int32_t page_size;    /* P: 0 (contiguous) or 32 (paged) */
  int32_t num_pages;    /* NP: pages in the pool of a paged cache (ignored when P == 0) */
} kvq_cache_desc;

/* Device pointers of one layer's cache (layout above).  k_res/v_res may be NULL
 * when residual == 0, k_sink/v_sink/sink_len when sink == 0, k_mode/v_mode when
 * hybrid == 0. */
typedef struct {
  uint8_t* k_codes;
  uint8_t* v_codes;
  uint32_t* k_params;
  uint32_t* v_params;
  uint16_t* k_res; /* fp16 bits */
  uint16_t* v_res;
  int32_t* packed_len;
  int32_t* res_len;
  int32_t* res_head;
  uint32_t* err_word;
  uint16_t* k_sink; /* fp16 bits */
  uint16_t* v_sink;
  int32_t* sink_len;
  uint8_t* k_mode; /* mode bytes [B][Hkv][cap] */
  uint8_t* v_mode;
  int32_t* block_table; /* [B][cap / 32], paged caches only */
} kvq_cache_view;

/* Which array kvq_cache_bytes sizes (each of K and V has one of each). */
#define KVQ_ARRAY_CODES 0
#define KVQ_ARRAY_PARAMS 1
#define KVQ_ARRAY_RESIDUAL 2
#define KVQ_ARRAY_SINK 3
#define KVQ_ARRAY_MODE 4

/* Bytes of one array of the layout (for K or for V; allocate twice).  For a
 * paged cache the codes, params and mode arrays are sized for the page pool.
 * Returns 0 for an invalid desc or `which`. */
size_t kvq_cache_bytes(const kvq_cache_desc* desc, int which);

/* Bytes of scratch kvq_decode_attention and kvq_decode_step need for num_q_heads
 * query heads on the current device.  Returns 0 for an invalid desc. */
size_t kvq_decode_workspace_bytes(const kvq_cache_desc* desc, int32_t num_q_heads);

/* Quantize and pack a prefill (Q1-Q6; BitDecoding page section 2.1 for the rule,
 * section 2.2 for the residual split, section 3.1 for the warp-shuffle kernel;
 * InnerQ page section 2.1 for the grouping along head_dim).
 *   k, v      fp16 device [B][Hkv][Lmax][d], row-major.
 *   seq_lens  int32 device [B], 0 <= seq_lens[b] <= Lmax.
 *   Lmax      host int, >= 0.
 * For each sequence b with L = seq_lens[b], split as in Q6: the first min(S, L)
 * tokens are copied to the sink (InnerQ page section 2.3), the next ones become
 * codes and params in slots [0, ...), the last min(Nr, ...) are copied to the
 * residual ring; packed_len[b], res_len[b], res_head[b] = 0 and (S > 0)
 * sink_len[b] are written.  A hybrid cache quantizes by H1-H3 (InnerQ page
 * section 2.2) and writes each packed row's mode byte.
 * A sequence with more than cap packed tokens sets KVQ_ERRBIT_CAPACITY and stores
 * only the first cap (packed_len[b] = cap).  Asynchronous on `stream`. */
kvq_status kvq_quantize_pack(const kvq_cache_desc* desc, const kvq_cache_view* view,
                             const void* k, const void* v, const int32_t* seq_lens,
                             int32_t Lmax, void* stream);

/* kvq_quantize_pack reading K and V in the layout the prefill produced them, in
 * the same single pass (the quantizer reads each group straight from the
 * producer's memory; nothing is transposed or copied first).  Same rule,
 * split, outputs, errors and asynchrony as kvq_quantize_pack; only the input
 * addressing differs:
 *   element j of head_dim of token t, KV head h, sequence b of k (and of v) is
 *   k[b * stride_b + h * stride_h + t * stride_t + j]   (fp16, strides in elements),
 *   read for t < seq_lens[b] <= Lmax.
 * Head-major [B][Hkv][Lmax][d]: (Hkv*Lmax*d, Lmax*d, d) (kvq_quantize_pack).
 * Token-major [B][L][Hkv][d]: (L*Hkv*d, d, Hkv*d).
 * A fused QKV projection output [B][L][(Hq + 2*Hkv)*d] (queries, then keys, then
 * values of each token): k = base + Hq*d, v = base + (Hq + Hkv)*d, strides
 * (L*W, d, W) with W = (Hq + 2*Hkv)*d.
 * The strides must be non-negative multiples of 8 (KVQ_ERR_MISALIGNED
 * otherwise), k and v 16-byte aligned. */
kvq_status kvq_quantize_pack_strided(const kvq_cache_desc* desc, const kvq_cache_view* view,
                                     const void* k, const void* v, const int32_t* seq_lens,
                                     int32_t Lmax, int64_t stride_b, int64_t stride_h,
                                     int64_t stride_t, void* stream);

/* Append one decode token per sequence (InnerQ page section 2.3, sliding recent
 * window).
 *   k_new, v_new  fp16 device [B][Hkv][d].
 * Per sequence: if res_len == Nr, the oldest residual token (ring slot res_head)
 * is quantized by Q1-Q5 into packed slot packed_len (which then grows by one)
 * and the new token takes its ring slot (res_head advances); otherwise the new
 * token goes to slot (res_head + res_len) % Nr and res_len grows.  With Nr == 0
 * the new token is packed directly (a hybrid cache by H1-H3, with its mode
 * byte).  The sink is never written: it stays as the
 * prefill left it.  A full packed cache sets KVQ_ERRBIT_CAPACITY and leaves that
 * sequence unchanged.  Asynchronous. */
kvq_status kvq_append(const kvq_cache_desc* desc, const kvq_cache_view* view,
                      const void* k_new, const void* v_new, void* stream);

/* Output element type of the decode calls (their `flags`): fp16 by default,
 * fp32 with KVQ_OUT_F32.  Both are rounded once from the fp32 result; fp16
 * rounding alone moves an output of magnitude 4 or more by up to 2^-9 * |O|. */
#define KVQ_OUT_F32 2u

/* Decode attention (BitDecoding page sections 2.2-2.3; InnerQ page section 3.1).
 *   q          fp16 device [B][Hq][d]; query head hq uses KV head hq / (Hq / Hkv).
 *   out        device [B][Hq][d], fp16 (or fp32 with KVQ_OUT_F32):
 *              softmax(q K^T / sqrt(d)) V over the sink, the packed tokens
 *              (dequantized as min + code * scale) and the residual.
 *   workspace  device scratch of ws_bytes >= kvq_decode_workspace_bytes(desc, Hq),
 *              16-byte aligned, zeroed before its first use.  Each completed call
 *              leaves it ready for the next call with the same batch, KV heads,
 *              head_dim and Hq (its counters and accumulators back at zero), so
 *              it is zeroed once, not per call; zero it again before a call with
 *              another shape and after a call that reported KVQ_ERR_TIMEOUT.
 *              One workspace serves one call at a time.
 *   flags      0 or KVQ_OUT_F32; other bits return KVQ_ERR_INVALID_ARG.
 * A sequence with no tokens gets a zero output and sets KVQ_ERRBIT_EMPTY.
 * Asynchronous; lengths are read on the device. */
kvq_status kvq_decode_attention(const kvq_cache_desc* desc, const kvq_cache_view* view,
                                const void* q, int32_t num_q_heads, void* out,
                                void* workspace, size_t ws_bytes, uint32_t flags, void* stream);

/* One decode step of the serving loop: kvq_append(k_new, v_new) and then
 * kvq_decode_attention(q) over the cache as it is after the append (InnerQ page
 * section 2.3 for the window, BitDecoding page sections 2.2-2.3 for the
 * attention; fusing the two is this library's addition).
 *   q, out, workspace, ws_bytes, num_q_heads  as for kvq_decode_attention (the
 *              workspace size from kvq_decode_workspace_bytes covers this call).
 *   k_new, v_new  fp16 device [B][Hkv][d], as for kvq_append.
 * The cache bytes, counters and error bits afterwards are exactly those of the
 * two calls; the output equals the two calls' within rounding (the token packed
 * by this step is attended in fp32 from its codes rather than on the tensor
 * cores).  With head_dim 128 and at most 4 query heads per KV head this is one
 * kernel launch: the packed splits read only rows written before the step, the
 * split of each head that takes its fp16 rows (a split of its own, or in a
 * grid of several waves the last packed split) does the append's writes and
 * attends over the new and the packed token, and the counters move when the
 * last head of a sequence finishes.  Other shapes launch the append and the decode kernels in turn.  A
 * sequence whose packed cache is full is left unchanged, sets
 * KVQ_ERRBIT_CAPACITY and is attended as it was.
 *   flags      0, or KVQ_STEP_EARLY_CACHE_READ: the caller states that the
 *              kernel enqueued on `stream` just before this call does not write
 *              this cache (any array of its view, counters included) -- in a serving loop
 *              it computes q, k_new and v_new, and the cache was last written by
 *              this layer's previous step.  The step (launched as a programmatic
 *              dependent of that kernel) then reads the counters and cuts its
 *              ranges before it waits for that kernel, and starts its copies the
 *              moment the wait returns; q, k_new and v_new are read, and anything
 *              is written, only after the wait.
 *              Without the flag nothing is read before the wait.  KVQ_OUT_F32
 *              may be or'ed in (fp32 out).  Other bits return KVQ_ERR_INVALID_ARG.
 * Asynchronous. */
#define KVQ_STEP_EARLY_CACHE_READ 1u
kvq_status kvq_decode_step(const kvq_cache_desc* desc, const kvq_cache_view* view,
                           const void* q, int32_t num_q_heads, const void* k_new,
                           const void* v_new, void* out, void* workspace, size_t ws_bytes,
                           uint32_t flags, void* stream);

/* Bytes of device staging kvq_decode_step_host needs: the packed input
 * [q | k_new | v_new] (fp16, in that order, no padding) and, at the next
 * 256-byte boundary, out (room for an fp32 out).  Returns 0 for an invalid desc
 * or head count. */
size_t kvq_step_io_bytes(const kvq_cache_desc* desc, int32_t num_q_heads);

/* kvq_decode_step with its inputs and output in host memory (no passage of the
 * pages corresponds to it; it is this library's serving-loop entry point).
 *   in_host    host [q (B*Hq*d) | k_new (B*Hkv*d) | v_new (B*Hkv*d)] fp16, the
 *              layouts of kvq_decode_step, contiguous in that order.
 *   out_host   host [B][Hq][d], fp16 (fp32 with KVQ_OUT_F32 in flags).
 *   dev_io     device staging of dev_io_bytes >= kvq_step_io_bytes(desc, Hq),
 *              256-byte aligned, owned by the caller.
 * Enqueues on `stream`: one host-to-device copy of the input block, the step
 * (as kvq_decode_step with the same workspace and flags, less
 * KVQ_STEP_EARLY_CACHE_READ: the step follows the copy, so there is nothing to
 * overlap), and one device-to-host copy of out.  Asynchronous when the host
 * buffers are pinned (page-locked), in which case they must stay valid until
 * the stream reaches the copies; with pageable memory the copies are
 * synchronous.  Argument errors return before anything is enqueued.
 *   flags | KVQ_STEP_HOST_MAPPED: in_host and out_host are page-locked host
 *              memory the device addresses with the same pointer (cudaHostAlloc,
 *              or registered with mapping; checked with cudaPointerGetAttributes,
 *              KVQ_ERR_INVALID_ARG otherwise).  No copy is enqueued: the step
 *              kernel reads the input block and writes out in place over the
 *              host link (NVLink-C2C on Grace hosts), dev_io is unused (may be
 *              NULL), and KVQ_STEP_EARLY_CACHE_READ keeps its meaning (the
 *              kernel before this call is the one it overlaps).  The buffers
 *              must stay valid until the step completes. */
#define KVQ_STEP_HOST_MAPPED 4u
kvq_status kvq_decode_step_host(const kvq_cache_desc* desc, const kvq_cache_view* view,
                                const void* in_host, int32_t num_q_heads, void* out_host,
                                void* dev_io, size_t dev_io_bytes, void* workspace,
                                size_t ws_bytes, uint32_t flags, void* stream);

/* Size of the device scratch array behind kvq_decode_attention_noalloc (8 MiB). */
#define KVQ_NOALLOC_SCRATCH_BYTES (8u << 20)

/* Decode attention without any caller-provided scratch, for callers that cannot
 * allocate device memory when they decode (a runtime that forbids cudaMalloc in
 * its serving loop, an allocator the caller does not own, memory fixed at start
 * up).  No passage of the pages corresponds to this call; it is an addition of
 * this library.
 * Same arguments (flags included), output and error bits as
 * kvq_decode_attention, minus the workspace: the split partials go to one static device array of
 * KVQ_NOALLOC_SCRATCH_BYTES that every GPU loading the library holds until the
 * process exits.  Returns KVQ_ERR_UNSUPPORTED when the decode would need more
 * than that (kvq_decode_workspace_bytes(desc, num_q_heads) > the maximum) and
 * KVQ_ERR_INVALID_ARG for an invalid description or head count.  Allocates
 * nothing.  The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current); make that first call before
 * any stream capture.  All calls share the array and it keeps the last call's
 * contents (its counters back at zero).  The first call on a device, a call whose
 * cache shape or head count differs from the previous call's there, and the
 * first call after kvq_read_error reported KVQ_ERR_TIMEOUT first clear the
 * array's counters and accumulators with cudaMemsetAsync on `stream`, so that
 * clear is ordered before the decode on the caller's own stream.  Calls whose
 * kernels overlap on the GPU race: keep them on one stream or order the
 * streams. */
kvq_status kvq_decode_attention_noalloc(const kvq_cache_desc* desc, const kvq_cache_view* view,
                                        const void* q, int32_t num_q_heads, void* out,
                                        uint32_t flags, void* stream);

/* Synchronize `stream`, copy *err_word to *word_out (may be NULL), clear it, and
 * return KVQ_OK if it was 0, else the status of its lowest set bit. */
kvq_status kvq_read_error(const kvq_cache_view* view, uint32_t* word_out, void* stream);

/* Static text for a status code. */
const char* kvq_status_string(kvq_status status);

/* Library version as 10000 * major + 100 * minor + patch. */
int32_t kvq_version(void); /* 160: two-part weights in the tensor-core MMAs, MMA rounding hook;
                              150: timeout testing hook, cached tensor maps; 140: paged caches;
                              130: 3-bit; 120: hybrid; 110: sink, fp32 out */

/* Testing hook, for checking the bounded-wait error path without faulting the
 * GPU (no passage of the pages corresponds to it).  With limit_us > 0, every
 * later tensor-core decode call (kvq_decode_attention, kvq_decode_step with
 * head_dim 128 and at most 4 query heads per KV head, and the calls built on
 * them) arms the barrier of the first tile of split 0 of (sequence 0, KV head 0)
 * for 16 bytes more than that tile's copies deliver, and gives every bounded
 * wait a limit of limit_us microseconds instead of one second.  All copies still
 * complete, so nothing is in flight when that CTA gives up: it sets
 * KVQ_ERRBIT_TIMEOUT, contributes nothing to its head's output (which is then
 * wrong for that head) and returns; the call's other results are unaffected.
 * limit_us = 0 (the default) restores normal behaviour.  Process-wide; not for
 * production use. */
void kvq_testing_wait_fault(uint32_t limit_us);

/* Testing hook (no passage of the pages corresponds to it): exhaustive checks,
 * on the current device, of the quantizer's fast arithmetic against the IEEE
 * operations it replaces.  div_mismatches[2i], [2i + 1] (i = 0, 1, 2 for the
 * divisors 2^b - 1 = 15, 7, 3): how many non-negative finite floats d give a
 * quotient d / (2^b - 1) other than the IEEE divide's, in all and in the
 * quantizer's domain (0 and the differences of fp16 values, 2^-24 .. 131008);
 * rcp_worst_rel: the largest relative error of the reciprocal used for the codes,
 * over every positive finite fp16 scale.  Synchronous (legacy default stream). */
kvq_status kvq_testing_check_arithmetic(uint64_t* div_mismatches, double* rcp_worst_rel);

/* Testing hook (no passage of the pages corresponds to it): how the tensor
 * cores round the f16 -> f32 MMA that the decode kernel's contractions use.
 * Runs eight fixed cases of one mma.sync m16n8k16, each C = c0 plus one product
 * `big` and fifteen products `small` (small in units of the float spacing at 1,
 * 2^-23): (c0, big, small) = (0, 1, 1/2), (0, 1, 1/4), (0, 1, 1/8),
 * (0, 1, 1/16), (1, 0, 1/2), (1, 0, 1/4), (0, 1, -1/2), (0, 1, -1/4), and
 * writes the first n (<= 8) results to the host array out.  Synchronous (legacy
 * default stream).  KVQ_ERR_INVALID_ARG for a null out or n outside 0..8. */
kvq_status kvq_testing_mma_rounding(float* out, int32_t n);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H_ */
