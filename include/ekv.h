/*
 * ekv.h — C ABI of the mixed-precision quantized KV-cache decode library (GB300, sm_103a).
 *
 * The library keeps, per layer, a paged KV cache whose pages carry their own
 * K bit-width (2, 4, 8 or 16 bits), an FP16 ring of each layer's newest 64 K
 * vectors, and a per-layer tier controller.  It implements:
 *
 *   ekv_append       quantize-and-append of new K/V tokens into the paged cache
 *   ekv_decode_attn  single-token GQA decode attention over the mixed-format pages
 *   ekv_append_decode_attn  both of them as one launch (the decode step of a layer)
 *   ekv_canary_kl    the canary: KL between FP16 attention over the ring and its
 *                    2/4/8-bit quantize-dequantize copies (ekv_canary_kl_layers:
 *                    every layer of a step in one launch)
 *   ekv_tier_update  EMA of the canary readings and lowest-bit-under-tau tier pick
 * and, around them: the KIVI-style asymmetric quantizer as a per-handle option
 * (ekv_config.quantizer), and the static-artifact mode's frozen clipping
 * thresholds (ekv_set_clip), percentile select (ekv_abs_percentile) and AutoK
 * layer allocator (ekv_autok).
 *
 * Sources of the operations (page title, section):
 *   - "EchoKV: watching a language model decide its own precision":
 *     "How EchoKV works" (ring written before quantization, tier vector routes
 *     future K blocks), "Do we store the whole cache in FP16? — No." (64-key
 *     FP16 ring, K only), "What happens to old blocks when a layer changes
 *     tier?" (admit-time bits, forward-only), "Show the math" (KL, EMA, pick).
 *   - "Behavior-Guided KV-Cache Quantization": "K/V Role-Aware Low-Bit
 *     Quantization" (K per channel, V per token, symmetric), "Storage savings,
 *     with a conditional speed trade-off" (packed low-bit storage, GQA head
 *     mapping, decode kernels).
 *   - "KV-Kaizen": "Three Non-Eviction Compression Axes" (symmetric uniform
 *     quantization, b in {2,4,8,16}).
 *
 * Conventions for every entry point:
 *   - Return value is an ekv_status; nothing throws across the ABI.
 *   - "dev" pointers are CUDA device pointers, "host" pointers are host memory.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Work is enqueued asynchronously on it unless the comment says "syncs".
 *   - Caller-owned buffers (Q, K, V, O, seq_slots, delta) must stay valid
 *     until the enqueued work completes.  The library owns everything else.
 *   - Errors found on the host (bad arguments) return at once and enqueue
 *     nothing.  Errors found on the device (a page pool running empty, a
 *     sequence growing past max_seq_len, a corrupt page entry) are recorded in
 *     a device error word; ekv_sync returns and clears it.
 *   - A handle is not thread-safe; calls on one handle must be serialized,
 *     and the work of one layer must not run concurrently on two streams.
 *   - Inputs must be finite fp16 values.
 */
#ifndef EKV_H
#define EKV_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define EKV_API __attribute__((visibility("default")))
#else
#define EKV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum ekv_status {
  EKV_OK = 0,
  EKV_EINVAL = 1,         /* invalid argument; nothing was enqueued                     */
  EKV_ENOMEM = 2,         /* allocation failed, or a page pool ran empty on the device  */
  EKV_ECUDA = 3,          /* a CUDA call or kernel launch failed                        */
  EKV_ETIMEOUT = 4,       /* a bounded device-side wait gave up                         */
  EKV_EUNSUPPORTED = 5,   /* valid request outside what this library implements         */
  EKV_ESTATE = 6          /* device detected an inconsistent state (capacity, entries)  */
} ekv_status;

#define EKV_BLOCK_TOKENS 16 /* tokens per page                                          */
#define EKV_RING_LEN 64     /* K vectors kept in each FP16 ring                          */

/* Page formats: index = kcode * 4 + vcode, code 0..3 <-> 2, 4, 8, 16 bits. */
#define EKV_NUM_FORMATS 16
#define EKV_FORMAT(kbits_code, vbits_code) ((kbits_code) * 4 + (vbits_code))

typedef struct ekv_cache ekv_cache;

typedef struct ekv_config {
  int32_t num_layers;
  int32_t max_seqs;        /* sequence slots 0 .. max_seqs-1                           */
  int32_t num_q_heads;     /* Hq; must be a multiple of num_kv_heads                   */
  int32_t num_kv_heads;    /* Hkv; query head h reads KV head h / (Hq / Hkv)           */
  int32_t head_dim;        /* 64 or 128                                                */
  int32_t max_seq_len;     /* tokens per sequence per layer (sets the block-table width) */
  int64_t pool_pages[EKV_NUM_FORMATS]; /* page capacity per format (0 = no pool)     */
  float softmax_scale;     /* 0 -> 1/sqrt(head_dim)                                    */
  float ema_alpha;         /* EMA weight of a new canary reading                        */
  float tau;               /* divergence budget of the tier pick                        */
  /* Controller variants ("EchoKV: watching a language model decide its own
   * precision": "The tau(L) scaling", and the hysteresis / multi-firing vote it
   * proposes against drift).  Zero turns each off. */
  int32_t tau_ctx0;        /* > 0: budget tau * sqrt(L / tau_ctx0), L = mean cached
                              length of the layer's sequences with tokens          */
  float hysteresis;        /* in [0, 1): picking fewer bits than the current tier
                              needs ema_b < budget * (1 - hysteresis)                */
  int32_t vote;            /* >= 2: a tier changes only after that many consecutive
                              firings picked the same new tier                      */
  /* Quantizer of every page and of the canary: EKV_QUANT_SYMMETRIC (0, the
   * default) or EKV_QUANT_ASYMMETRIC (1, KIVI-style: "EchoKV: watching a
   * language model decide its own precision", "Show the math" names it for the
   * canary and "Upstreaming into vLLM" for the cache).  Per group (K: a
   * channel over a block's 16 tokens, V: a token's d channels; the canary: a
   * channel over a 16-row group of the ring): lo, hi = min, max;
   * s = fp16_rne((hi - lo) / (2^b - 1)) (fp32 subtraction and division);
   * z = lo; u = clamp(rne((x - z) / s), 0, 2^b - 1) (0 if s = 0); the value
   * read back is u * s + z.  Codes are stored unsigned; each quantized part
   * adds one fp16 zero point per group after its scales. */
  int32_t quantizer;
  /* Device allocator.  NULL -> cudaMalloc/cudaFree.  Called only inside
   * ekv_create/ekv_destroy; must return 16-byte aligned memory (else
   * ekv_create fails with EKV_ENOMEM). */
  void* (*dev_alloc)(size_t bytes, void* ctx);
  void (*dev_free)(void* ptr, void* ctx);
  void* alloc_ctx;
} ekv_config;

#define EKV_QUANT_SYMMETRIC 0
#define EKV_QUANT_ASYMMETRIC 1

/* Human-readable name of a status code (static string, never NULL). */
EKV_API const char* ekv_status_string(int status);

/* Bytes of one page of format (k_bits, v_bits) at head_dim d; -1 if invalid.
 * Layout (one layer, one sequence, one KV head, 16 token slots):
 *   K part  k_bits < 16: codes [16][d*k_bits/8], then per-channel scales [d] fp16
 *           k_bits = 16: raw fp16 [16][d]
 *   V part  v_bits < 16: codes [16][d*v_bits/8], then per-token scales [16] fp16
 *           v_bits = 16: raw fp16 [16][d]
 * Codes are offset binary (q + 2^(b-1)), packed along channels, least
 * significant bits first: channel c sits in byte c*b/8 at bit (c*b)%8. */
EKV_API int32_t ekv_page_bytes(int32_t k_bits, int32_t v_bits, int32_t head_dim);
/* The same for a quantizer (EKV_QUANT_*): the asymmetric one adds a zero-point
 * row after each quantized part's scales (K: [d] fp16, same order as the K
 * scales; V: [16] fp16).  -1 for an invalid argument. */
EKV_API int32_t ekv_page_bytes_q(int32_t k_bits, int32_t v_bits, int32_t head_dim,
                                 int32_t quantizer);

/* Create a cache.  k_bits_init[num_layers] (host): each layer's starting K tier
 * (2, 4, 8 or 16).  v_bits[num_layers] (host): each layer's fixed V width.
 * Allocates every pool, table, ring and scratch buffer up front and zeroes
 * them; syncs the device.  *out receives the handle. */
EKV_API int ekv_create(const ekv_config* cfg, const uint8_t* k_bits_init, const uint8_t* v_bits,
               ekv_cache** out);

/* Free everything ekv_create allocated (syncs the device).  NULL is a no-op. */
EKV_API int ekv_destroy(ekv_cache* cache);

/* Return every page of sequence slot `seq_slot` (all layers) to its pool and
 * set its length to 0. */
EKV_API int ekv_seq_reset(ekv_cache* cache, int32_t seq_slot, void* stream);

/* Append n_new tokens to each listed sequence of one layer.
 *   seq_slots [n_seqs] int32 dev — distinct slot ids
 *   k, v      [n_seqs][n_new][Hkv][d] fp16 dev — the new tokens, in order
 * Per token: the K vector enters the layer's FP16 ring; a page is allocated
 * at the layer's current tier when the token opens a block (its K bits never
 * change afterwards); V is quantized per token (absmax over d channels) into
 * the page; K is kept raw in the block's staging rows until the 16th token
 * seals the block, which quantizes each channel over the 16 tokens.
 * Quantizer: s = fp16_rne(absmax / qmax) with qmax = 2^(b-1)-1,
 * q = clamp(rne(x / s), -qmax, qmax) (q = 0 if s = 0).  n_new >= 1 (prefill
 * in one call is allowed).  A pool running empty sets EKV_ENOMEM on the
 * device; that sequence must then be reset. */
EKV_API int ekv_append(ekv_cache* cache, int32_t layer, int32_t n_seqs, const int32_t* seq_slots,
               int32_t n_new, const void* k, const void* v, void* stream);

/* Decode attention of one layer.
 *   q [n_seqs][Hq][d] fp16 dev;  o [n_seqs][Hq][d] fp16 dev (written)
 * o_h = sum_t softmax_t(scale * q_h . khat_t) vhat_t over every cached token
 * of the sequence, with KV head h / (Hq/Hkv); khat/vhat are the dequantized
 * page values (raw fp16 for rows of a still-open block).  fp32 accumulation,
 * split over the context with a log-sum-exp merge; o rounded to fp16 (RNE).
 * A sequence with no tokens gets o = 0.  Requires Hq/Hkv <= 8. */
EKV_API int ekv_decode_attn(ekv_cache* cache, int32_t layer, int32_t n_seqs, const int32_t* seq_slots,
                    const void* q, void* o, void* stream);

/* One decode step of one layer in one launch: ekv_append with n_new = 1
 * followed by ekv_decode_attn, with the same results (pages, staging rows,
 * ring, length and o; o's fp32 summation order may differ, as it does between
 * any two launches).  The append work of each (sequence, KV head) runs inside
 * the attention launch, on the split that holds the sequence's last block,
 * while the other splits stream their pages, so the step pays one launch and
 * no separate chain of append memory round trips.  The pages define the two
 * steps ("How EchoKV works": the step's K enters the ring and the paged cache
 * before attention reads it); fusing them is this library's choice.
 *   k, v [n_seqs][Hkv][d] fp16 dev — the new token of each sequence
 *   q, o as ekv_decode_attn.  All four 16-byte aligned.
 *   flags   0, EKV_AFTER_OTHER_LAYER or EKV_AFTER_PRODUCER; either lets the
 *           launch start before the work queued just before it on `stream`
 *           has finished (programmatic dependent launch): it takes the SMs
 *           that work frees and streams this layer's pages meanwhile.
 *           EKV_AFTER_OTHER_LAYER: the caller states that the previous work is
 *           an ekv_append_decode_attn of another layer of the same handle and
 *           writes none of this call's seq_slots, k, v and q.  The launch reads
 *           them early and waits for that work only before writing o or the
 *           handle's shared split scratch.
 *           EKV_AFTER_PRODUCER: the previous work may write k, v and q (as the
 *           projections feeding this layer do in a model), but writes none of
 *           seq_slots and no state of this handle's layer `layer` (it is not an
 *           append to this layer).  Before that work finishes the launch reads
 *           only seq_slots and this layer's lengths, page table and pages; it
 *           waits before its first read of q, k or v and before any write.
 *           Both bits: as EKV_AFTER_PRODUCER.  Any other bit: EKV_EINVAL.
 *           (A decode-attention launch lets its own programmatic dependents
 *           start once every CTA has passed its wait for the work before it:
 *           with EKV_AFTER_PRODUCER near its start, otherwise before it writes
 *           o.  Work launched after it with programmatic stream serialization
 *           must wait for it (griddepcontrol.wait, i.e.
 *           cudaGridDependencySynchronize) before reading o or any state of this
 *           handle.  Work launched without that attribute sees ordinary stream
 *           order.)
 * Errors as the two calls: EKV_ENOMEM on the device when a pool runs empty;
 * a sequence whose table is full gets EKV_ESTATE, no append, and attention
 * over its old tokens. */
#define EKV_AFTER_OTHER_LAYER 1
#define EKV_AFTER_PRODUCER 2
EKV_API int ekv_append_decode_attn(ekv_cache* cache, int32_t layer, int32_t n_seqs,
                                   const int32_t* seq_slots, const void* k, const void* v,
                                   const void* q, void* o, int32_t flags, void* stream);

/* Allocation-free decode attention.  The pages have no counterpart of this
 * entry point; it exists for callers that cannot allocate device memory where
 * they run attention (a process that reserves all device memory at start-up
 * and forbids later cudaMalloc, or code that cannot reach the allocator the
 * handle was created with).
 * Same arguments, kernel, split schedule and results as ekv_decode_attn, but
 * the split-K scratch (partial numerators, (max, sum) pairs and merge
 * tickets) comes from one static device array of EKV_NOALLOC_SCRATCH_BYTES
 * built into the library instead of the handle's scratch.  It calls no
 * allocator.
 *   - Limit: n_seqs * Hkv * splits * 8 * (d + 2) * 4 bytes of partials plus
 *     n_seqs * Hkv * 17 * 4 bytes of tickets (each part 256-byte aligned) must fit
 *     in EKV_NOALLOC_SCRATCH_BYTES; larger requests return EKV_EINVAL and
 *     enqueue nothing.  splits is the split count ekv_decode_attn uses for
 *     n_seqs on this handle.
 *   - Every GPU that loads the library holds the array until the process
 *     exits.  The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.  The address is kept for the life of the
 *     process: after cudaDeviceReset (or any other teardown of the device's
 *     primary context) it is stale, so do not call this entry point again in
 *     that process.
 *   - All calls share the array and it keeps the last call's contents; each
 *     call clears the tickets it uses (cudaMemsetAsync on `stream`) before
 *     launching.  Calls that overlap on the GPU race on the array: serialize
 *     them. */
#define EKV_NOALLOC_SCRATCH_BYTES (4u << 20)
EKV_API int ekv_decode_attn_noalloc(ekv_cache* cache, int32_t layer, int32_t n_seqs,
                                    const int32_t* seq_slots, const void* q, void* o,
                                    void* stream);

/* Canary of one layer: for every listed sequence and query head, the KL
 * divergence KL(softmax(scale q W^T) || softmax(scale q quant_b(W)^T)) over
 * the ring window W (the newest min(len, 64) K vectors, oldest first), for
 * b = 2, 4, 8, where quant_b quantizes each channel over consecutive 16-row
 * groups of W starting at the oldest row.  The mean over all n_seqs*Hq
 * queries is stored as the layer's reading delta[layer][0..2] (internal) and,
 * if delta_out (dev float[3]) is not NULL, copied there. */
EKV_API int ekv_canary_kl(ekv_cache* cache, int32_t layer, int32_t n_seqs, const int32_t* seq_slots,
                  const void* q, float* delta_out, void* stream);

/* The canary of layers first_layer .. first_layer+n_layers-1 in one launch, with
 * the same readings as n_layers calls of ekv_canary_kl.  Layer first_layer+i
 * reads its queries [n_seqs][Hq][d] at q + i * q_layer_stride (fp16 elements,
 * >= n_seqs*Hq*d when n_layers > 1) and, if delta_out (dev float[n_layers][3])
 * is not NULL, writes its readings to delta_out[i].  A decode step that fires
 * the canary calls it once, after every layer's append (a layer's ring and
 * queries are final then): one launch instead of one per layer. */
EKV_API int ekv_canary_kl_layers(ekv_cache* cache, int32_t first_layer, int32_t n_layers,
                                 int32_t n_seqs, const int32_t* seq_slots, const void* q,
                                 int64_t q_layer_stride, float* delta_out, void* stream);

/* Controller update for every layer whose layer_mask entry is nonzero
 * (layer_mask dev uint8[num_layers], NULL = all layers):
 *   ema = first reading ? delta : (1-alpha)*ema + alpha*delta   (fp32, unfused)
 *   budget = tau, or with tau_ctx0 > 0 and sequences holding tokens:
 *            tau * sqrt(L / tau_ctx0), L = sum of their lengths / their count
 *            (fp32: one rounding per division, square root and product)
 *   pick = min{ b in {2,4,8} : ema_b < (b < tier ? budget*(1-hysteresis) : budget) },
 *          else 8
 *   tier = pick once `vote` consecutive firings picked it (vote <= 1: at once);
 *          a firing that picks the current tier resets the count.
 * delta (dev float[num_layers][3]) NULL = the readings stored by ekv_canary_kl.
 * freeze != 0 leaves every EMA and tier unchanged.  A new tier governs pages
 * allocated by later appends only. */
EKV_API int ekv_tier_update(ekv_cache* cache, const float* delta, const uint8_t* layer_mask,
                    int32_t freeze, void* stream);

/* Overwrite the tiers (host uint8[num_layers], each 2, 4, 8 or 16). */
EKV_API int ekv_set_tiers(ekv_cache* cache, const uint8_t* tiers, void* stream);

/* ---- Static-artifact mode ("Behavior-Guided KV-Cache Quantization": the
 * framework's "Freeze & allocate" and "Online inference" stages, "Calibration
 * protocol", "Sensitivity-Driven Budget Allocation").  Offline calibration
 * freezes clipping thresholds (theta*) and per-layer bits (b*); online, the
 * cache is created with b* as its tiers, the thresholds are loaded, and the
 * controller is left unfired (read-only configuration). */

/* Clipping thresholds of one layer (host float arrays; syncs stream):
 *   k_clip [Hkv][d]  per (KV head, channel): caps each sealed K block's
 *                    per-channel absmax, m = min(absmax, c);
 *   v_clip [Hkv]     per KV head: caps each V token's absmax.
 * The quantizer is otherwise unchanged (s = fp16_rne(m / qmax), codes clamped
 * to +-qmax, so values beyond c take the end codes).  The canary quantizes the
 * ring with the same K thresholds.  NULL = no clipping (+inf) for that part;
 * every threshold must be > 0 (+inf allowed), else EKV_EINVAL and nothing
 * changes.  A handle with the asymmetric quantizer returns EKV_EUNSUPPORTED.  New thresholds govern pages sealed and V rows written afterwards;
 * pages already written keep their bytes.  A new handle has no clipping. */
EKV_API int ekv_set_clip(ekv_cache* cache, int32_t layer, const float* k_clip,
                         const float* v_clip, void* stream);
/* Read one layer's thresholds back (host outputs, either may be NULL; syncs). */
EKV_API int ekv_get_clip(ekv_cache* cache, int32_t layer, float* k_clip, float* v_clip,
                         void* stream);

/* Nearest-rank quantile of |x| per group (a calibration threshold):
 *   x       dev fp16, 2-byte aligned; group g's elements are
 *           x[r * row_stride + g * group_stride + i], r < n_rows, i < group_width
 *           (strides in elements; every addressed element must lie in the buffer)
 *   out     dev float[n_groups], 4-byte aligned
 *   scratch dev, 4-byte aligned, at least ekv_abs_percentile_scratch_bytes
 *           (n_groups) bytes (caller-owned; overwritten; one call at a time)
 * With the group's n = n_rows * group_width magnitudes sorted ascending, out[g]
 * is the one of 1-based rank max(1, ceil(q * n)) (q * n in fp64), so it is one
 * of the group's own values.  K thresholds of [T][Hkv][d] keys: n_rows = T,
 * row_stride = Hkv*d, n_groups = Hkv*d, group_stride = 1, group_width = 1.
 * V thresholds per head: n_groups = Hkv, group_stride = d, group_width = d.
 * Needs 0 <= q <= 1, n < 2^32 and finite inputs; else EKV_EINVAL (nothing enqueued). */
EKV_API int ekv_abs_percentile(const void* x, int64_t n_rows, int64_t row_stride,
                               int32_t n_groups, int64_t group_stride, int32_t group_width,
                               double q, float* out, void* scratch, int64_t scratch_bytes,
                               void* stream);
/* Scratch bytes ekv_abs_percentile needs for n_groups groups (host only). */
EKV_API int ekv_abs_percentile_scratch_bytes(int32_t n_groups, int64_t* out);

/* The sums behind the Value score of the calibration ("Behavior-Guided KV-Cache
 * Quantization", "K/V Role-Aware Low-Bit Quantization": Value candidates are
 * scored by the perturbation of the attention output): over n fp16 elements,
 * out[0] = sum (o_hat - o_ref)^2 and out[1] = sum o_ref^2, accumulated in fp64
 * (the order of the additions varies between calls).  o_hat, o_ref dev fp16
 * (2-byte aligned; may be NULL when n = 0); out host double[2]; scratch dev,
 * 8-byte aligned, 16 bytes (caller-owned, overwritten).  Syncs stream. */
EKV_API int ekv_output_error(const void* o_hat, const void* o_ref, int64_t n, double* out,
                             void* scratch, void* stream);

/* AutoK: the smallest number k of layers whose sensitivities, taken largest
 * first (equal values: lower index first), sum in fp64 to >= frac times the
 * sum of all n.  sensitivity host double[n] (finite, >= 0); 0 <= frac <= 1.
 * order_out (host int32[n], may be NULL) receives that order; *k_out = k.
 * The first k layers of the order are the ones to protect with more bits. */
EKV_API int ekv_autok(const double* sensitivity, int32_t n, double frac, int32_t* order_out,
                      int32_t* k_out);

/* Controller state (syncs stream).  Any output pointer may be NULL.
 *   tiers uint8[L], ema float[L][3], delta float[L][3], ema_valid int32[L] (host). */
EKV_API int ekv_get_state(ekv_cache* cache, uint8_t* tiers, float* ema, float* delta,
                  int32_t* ema_valid, void* stream);

/* Length (tokens) of one (layer, slot) (syncs stream). */
EKV_API int ekv_seq_len(ekv_cache* cache, int32_t layer, int32_t seq_slot, int32_t* out, void* stream);

/* Page-table entries of one (layer, slot, kv_head), in block order (syncs stream).
 * entry = (format << 28) | page index (negative as int32 for formats >= 8),
 * -1 = no page.  Writes min(cap, blocks
 * in use) entries to out (host) and the number of blocks in use to *n_out. */
EKV_API int ekv_block_table(ekv_cache* cache, int32_t layer, int32_t seq_slot, int32_t kv_head,
                    int32_t* out, int32_t cap, int32_t* n_out, void* stream);

/* Copy the raw bytes of pages first_block .. first_block+n_blocks-1 of one
 * (layer, slot, kv_head) into dst (dev), page i at dst + i*dst_stride
 * (dst_stride >= the largest page size of the layer).  Blocks without a page
 * are left untouched. */
EKV_API int ekv_read_pages(ekv_cache* cache, int32_t layer, int32_t seq_slot, int32_t kv_head,
                   int32_t first_block, int32_t n_blocks, void* dst, size_t dst_stride,
                   void* stream);

/* ---- Realized precision ("EchoKV: watching a language model decide its own
 * precision": the simulation's running "avg bits / element" and "memory saved
 * vs FP16", and "What the controller costs you in memory"; "KV-Kaizen":
 * "Action Space and Cost Model", c(a) = (d + d_R) * b bits per token against
 * the 16-bit cost C0).  What the cache of layers first_layer ..
 * first_layer+n_layers-1 holds over every sequence slot, one page per
 * (layer, slot, KV head, 16-token block):
 *   sealed_pages[f]  pages of format f whose block holds 16 tokens
 *   open_pages[f]    pages of format f of a sequence's still-open last block
 *   open_rows[f]     the tokens in those open blocks
 *   tokens           cached (layer, slot, KV head) tokens
 *   k_bits, v_bits   mean stored bits per cached K / V element: a page's K or V
 *                    width; K rows of an open block count 16 (they are held raw
 *                    in fp16 until the block seals)
 *   cost_vs_c0       (k_bits + v_bits) / 32: the code bits against C0 (no rank
 *                    truncation, d_R = 0)
 *   page_bytes       bytes of the pages in use, scales and zero points included
 *   fp16_bytes       the same tokens' K and V in fp16: tokens * head_dim * 4
 *   saved_vs_fp16    1 - page_bytes / fp16_bytes
 * Zero tokens give zero means.  Syncs stream; EKV_ESTATE if a block in use has
 * no page. */
typedef struct ekv_stats_t {
  int64_t sealed_pages[EKV_NUM_FORMATS];
  int64_t open_pages[EKV_NUM_FORMATS];
  int64_t open_rows[EKV_NUM_FORMATS];
  int64_t tokens;
  double k_bits;
  double v_bits;
  double cost_vs_c0;
  double page_bytes;
  double fp16_bytes;
  double saved_vs_fp16;
} ekv_stats_t;
EKV_API int ekv_stats(ekv_cache* cache, int32_t first_layer, int32_t n_layers, ekv_stats_t* out,
                      void* stream);

/* Free pages left in the pool of one format (syncs stream). */
EKV_API int ekv_pool_free(ekv_cache* cache, int32_t format, int64_t* out, void* stream);

/* Test hooks (off in a new handle).
 *   EKV_DEBUG_WAIT_EXPIRY  value != 0: every bounded device-side wait of decode
 *                          attention reports that it gave up once the copy it
 *                          waits for has landed.  The kernel then takes the path
 *                          of a real expiry (the warp stops taking pages, waits
 *                          for its copies still in flight, the launch returns and
 *                          ekv_sync reports EKV_ETIMEOUT; that launch's o is not
 *                          valid), with nothing left in flight and no stall.
 *                          0 restores normal waits.
 * Unknown knob: EKV_EINVAL. */
#define EKV_DEBUG_WAIT_EXPIRY 1
EKV_API int ekv_debug_set(ekv_cache* cache, int32_t knob, int64_t value);

/* Wait for the stream, then return and clear the device error word. */
EKV_API int ekv_sync(ekv_cache* cache, void* stream);

/* Controller checkpoint: tiers, EMA, EMA-valid flags, last readings.
 * ekv_state_size gives the blob size; save/load sync the stream. */
EKV_API int64_t ekv_state_size(ekv_cache* cache);
EKV_API int ekv_state_save(ekv_cache* cache, void* host_blob, int64_t bytes, void* stream);
EKV_API int ekv_state_load(ekv_cache* cache, const void* host_blob, int64_t bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* EKV_H */
