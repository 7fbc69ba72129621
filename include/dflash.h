/*
 * dflash.h -- C ABI of libdflash: one DFlash drafting-plus-acceptance round
 * on one NVIDIA GB300 GPU (sm_103a).
 *
 * A round ("DFlash原理深度剖析：块扩散如何用一次前向并行起草整块token", §三 第1-3步):
 *   dflash_fuse_inject  fuse the hidden states of 5 target layers into one
 *                       context feature per new position and inject it into
 *                       every draft layer's paged KV cache;
 *   dflash_draft_block  one forward of the draft transformer over a block of
 *                       S tokens [last verified token, (S-1) x mask] -> S-1
 *                       drafts (S = 16, the trained block, or smaller);
 *   dflash_accept_trim  given the target's own token per block position,
 *                       accept the longest matching prefix plus the bonus
 *                       token and trim the caches to the confirmed length.
 *
 * Conventions for every call:
 *   - Tensors are caller-owned DEVICE memory unless stated otherwise
 *     (bf16 = IEEE bfloat16, row-major, densely packed).
 *   - `stream` is a cudaStream_t passed as void*; work is enqueued on it and
 *     the call returns without synchronising (except where stated), so every
 *     call is legal inside CUDA stream capture.
 *   - The return value is a dflash_status.  No exception or abort crosses the
 *     ABI.  Host-side argument checks return an error and enqueue nothing.
 *     Device-side checks (slot ids, row counts, page capacity, NaN logits)
 *     never trap: they set bits in the handle's device status word, skip the
 *     offending work, and are reported by dflash_read_status.
 *   - Per-request state lives in "slots" (0 <= slot < max_slots).  A call on
 *     a batch takes a DEVICE int32 array `slots[batch]` mapping batch row b
 *     to its slot; a slot must not appear twice in one call.
 */
#ifndef DFLASH_H
#define DFLASH_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define DFLASH_API __attribute__((visibility("default")))
#else
#define DFLASH_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DFLASH_OK = 0,
  DFLASH_ERR_INVALID_ARG = 1, /* null pointer, negative size, batch > max_batch */
  DFLASH_ERR_SHAPE = 2,       /* shape the kernels do not support */
  DFLASH_ERR_CAPACITY = 3,    /* rows > max_rows, or the page pool is exhausted (device) */
  DFLASH_ERR_CUDA = 4,        /* a CUDA runtime call or kernel launch failed */
  DFLASH_ERR_DEVICE = 5,      /* a device-side check tripped; see dflash_read_status */
  DFLASH_ERR_WORKSPACE = 6,   /* workspace null, too small or not 256-byte aligned */
  DFLASH_ERR_RANGE = 7        /* dflash_create: a weight exceeds the f16 range (|w| > 65504) */
} dflash_status;

/* Device status word bits (dflash_read_status). */
#define DFLASH_DEV_TIMEOUT   0x01u /* a bounded wait inside a kernel gave up (2 s; the kernel then
                                       drains its copies in flight, frees its TMEM and returns) */
#define DFLASH_DEV_NAN       0x02u /* a NaN logit was skipped by the argmax */
#define DFLASH_DEV_PAGE      0x04u /* a page-table entry was out of range */
#define DFLASH_DEV_CAPACITY  0x08u /* page pool or per-slot page table full */
#define DFLASH_DEV_ARG       0x10u /* slot id or n_new out of range (the request is skipped: no
                                       cache entry written; its outputs are unspecified) */
#define DFLASH_DEV_RANGE     0x20u /* an f16 activation or cache entry exceeded 65504 (stored as
                                       +-65504, the largest finite f16; NaN stays NaN) */

/* Drafter shape and serving limits.
 * Supported: head_dim in {64,128}; intermediate a multiple of 64;
 * n_q_heads*head_dim and n_kv_heads*head_dim multiples of 128; hidden a
 * multiple of 128 and <= 8192; n_q_heads/n_kv_heads in {1, 2, 4, 8};
 * 2 <= block <= 16; page_size == 64; n_layers <= 8; max_batch <= 64.
 * Anything else makes dflash_workspace_bytes return 0 and dflash_create
 * return DFLASH_ERR_SHAPE. */
typedef struct dflash_config {
  int32_t hidden;             /* H */
  int32_t n_q_heads;          /* hq */
  int32_t n_kv_heads;         /* hkv */
  int32_t head_dim;           /* D */
  int32_t intermediate;       /* I (SwiGLU) */
  int32_t n_layers;           /* draft layers */
  int32_t vocab;              /* V (tied embedding / lm_head rows) */
  int32_t n_fused;            /* target layers fused (5) */
  int32_t block;              /* block size S: 1 verified token + S-1 masks.  16 is the
                                 trained size; a smaller S at inference ("DFlash：drafter
                                 的答案…", Results: a large training block generalises to
                                 smaller inference blocks) drafts S-1 tokens with the same
                                 kernels, rows S..15 of each request carried as padding */
  int32_t mask_id;            /* token id of the mask */
  int32_t page_size;          /* positions per KV page (64) */
  int32_t max_batch;          /* max requests per call */
  int32_t max_slots;          /* request slots */
  int32_t max_pages;          /* pages in the shared pool */
  int32_t max_pages_per_slot; /* page-table length per slot */
  int32_t max_rows;           /* max batch*rows_per_req of one dflash_fuse_inject */
  int32_t device;             /* CUDA device ordinal */
  float rms_eps;              /* RMSNorm epsilon (1e-6) */
  float rope_theta;           /* RoPE base */
  int32_t attn_impl;          /* block attention page loop: 0 by capacity (tensor cores from
                                 8 pages per split up), 1 warp MMAs, 2 tcgen05 */
  int32_t role;               /* 0: the drafter.  1: a target model of the same layer shape
                                 for dflash_verify_block / dflash_advance -- causal attention
                                 over its own paged cache, n_layers >= n_fused + 2, block 16,
                                 no fusion weights (fc, fc_norm may be null) */
  int32_t weight_fp8;         /* 1: every projection and the tied embedding held as FP8 E4M3
                                 with a float32 scale per output row (max |row| / 448, values
                                 rounded to nearest even, saturating), converted to f16 in the
                                 SM before each MMA, the scale applied in the epilogue; the
                                 fusion projection stays bf16.  Halves the weight bytes a round
                                 streams.  0: f16 (as below) */
} dflash_config;

/* Device pointers to the drafter weights, all bf16 and row-major; the arrays
 * of per-layer pointers are HOST arrays of n_layers entries.  They are read
 * only during dflash_create, which copies everything into the workspace:
 * matrices repacked into 128x64 tensor-core tiles (converted to f16, which
 * holds every bf16 weight of magnitude >= 2^-14 exactly and the smaller ones
 * to within 2^-25; the fusion projection stays bf16) and gains as float32.
 * The caller may free its buffers once dflash_create returns.  Activations,
 * the KV cache and the argmax logits are computed with f16 tensor-core
 * operands and fp32 accumulation; an activation beyond the f16 range is
 * saturated and sets DFLASH_DEV_RANGE.  With weight_fp8 = 0, a weight beyond
 * the f16 range makes dflash_create return DFLASH_ERR_RANGE (no handle is
 * created; weight_fp8 = 1 holds any finite weight through its row scale). */
typedef struct dflash_weights {
  const void* embed;             /* [V, H]  tied embedding and lm_head */
  const void* fc;                /* [H, n_fused*H] fusion projection (no bias) */
  const void* fc_norm;           /* [H]     fusion RMSNorm gain */
  const void* final_norm;        /* [H]     final RMSNorm gain */
  const void* const* in_norm;    /* [H]     input RMSNorm gain */
  const void* const* wqkv;       /* [(hq+2*hkv)*D, H] q rows, then k rows, then v rows */
  const void* const* q_norm;     /* [D]     per-head q RMSNorm gain */
  const void* const* k_norm;     /* [D]     per-head k RMSNorm gain */
  const void* const* wo;         /* [H, hq*D] */
  const void* const* post_norm;  /* [H]     post-attention RMSNorm gain */
  const void* const* w_gate_up;  /* [2*I, H] gate rows, then up rows */
  const void* const* w_down;     /* [H, I] */
} dflash_weights;

typedef struct dflash_handle dflash_handle;

/* Bytes of device workspace dflash_create needs for `cfg` (KV page pool,
 * page tables, activations, split-K and split-KV scratch, status word).
 * Returns 0 if cfg is invalid. */
DFLASH_API size_t dflash_workspace_bytes(const dflash_config* cfg);

/* Create a handle.  `workspace` is caller-allocated device memory of at least
 * dflash_workspace_bytes(cfg) bytes, 256-byte aligned, owned by the caller
 * and used exclusively by this handle until dflash_destroy.  Synchronises
 * the device (initialises the page pool, RoPE table and all slots to empty).
 * Not legal inside stream capture. */
DFLASH_API int dflash_create(const dflash_config* cfg, const dflash_weights* w, void* workspace,
                  size_t workspace_bytes, dflash_handle** out);
DFLASH_API int dflash_destroy(dflash_handle* h);

/* a1 + a2.  Feature fusion ("DFlash：drafter 的答案，早写在 target model 的隐层里",
 * 设计 — Feature Fusion: five target layers shallow->deep, concatenated, one
 * projection, RMSNorm) and KV injection (same page, 设计 — KV Injection: the
 * fused feature is projected by every draft layer's own K/V projections,
 * k-normed, rotated at its context positions and kept across rounds).
 *   feats  [batch, rows_per_req, n_fused, H] bf16; request b's new rows are
 *          its first n_new[b] rows (position order).
 *   n_new  DEVICE int32 [batch], 0 <= n_new[b] <= rows_per_req; rows are
 *          appended at positions ctx_len .. ctx_len+n_new-1 of the slot.
 * Prefill is one call with rows_per_req = prompt length.  In a round,
 * n_new is the previous round's accept_len (the same device buffer), which
 * keeps a captured round loop free of host reads.  Requires
 * batch*rows_per_req <= max_rows (else DFLASH_ERR_CAPACITY) and feats
 * 16-byte aligned (else DFLASH_ERR_INVALID_ARG); a target handle (role 1)
 * is refused with DFLASH_ERR_INVALID_ARG.  Every host-side refusal happens
 * before anything is enqueued: the slots' lengths and pages stay as they
 * were. */
DFLASH_API int dflash_fuse_inject(dflash_handle* h, const int32_t* slots, int32_t batch, const void* feats,
                       int32_t rows_per_req, const int32_t* n_new, void* stream);

/* a3-a6.  Embed the block [last_tok[b], mask x (S-1)] at positions
 * ctx_len .. ctx_len+S-1, run every draft layer once with non-causal
 * attention over [context KV ; block KV] ("DFlash原理深度剖析…", §二.1, §二.2),
 * apply the final RMSNorm and the tied lm_head, and write the argmax of
 * block rows 1..S-1 (ties -> lowest id; logits are never stored).
 *   last_tok DEVICE int32 [batch]; draft DEVICE int32 [batch, S-1] (out). */
DFLASH_API int dflash_draft_block(dflash_handle* h, const int32_t* slots, int32_t batch,
                       const int32_t* last_tok, int32_t* draft, void* stream);

/* a1-a6 in one call: exactly dflash_fuse_inject(slots, batch, feats,
 * rows_per_req, n_new) followed by dflash_draft_block(slots, batch, last_tok,
 * draft), with the K/V injection of the new rows computed inside each draft
 * layer's own QKV projection (the rows ride along as extra tokens of that
 * GEMM), so every layer's K/V weights are read once per round instead of
 * twice.  Used when rows_per_req <= 16 and batch*(16 + rows_per_req) <= 256;
 * otherwise it runs the two calls.  A drafter call: DFLASH_ERR_INVALID_ARG
 * on a target handle. */
DFLASH_API int dflash_draft_round(dflash_handle* h, const int32_t* slots, int32_t batch, const void* feats,
                                  int32_t rows_per_req, const int32_t* n_new, const int32_t* last_tok,
                                  int32_t* draft, void* stream);

/* a7.  Longest-prefix acceptance (cumulative product of matches,
 * "DFlash原理深度剖析…", §三 第3步).  draft [batch,S-1], target [batch,S] (the
 * target's token after each block position).  Outputs (DEVICE int32 [batch]):
 *   accept_len = accepted drafts + 1, in [1, S];
 *   bonus      = target[b][accept_len-1] (the next round's last verified token);
 *   ctx_len    = confirmed length = ctx_len_before_round + accept_len, the length
 *                both the draft and the target caches are trimmed to.
 * The draft cache never keeps block K/V, so trimming it only clamps the
 * slot's length to the confirmed one; the accept_len new features are
 * appended by the next dflash_fuse_inject. */
DFLASH_API int dflash_accept_trim(dflash_handle* h, const int32_t* slots, int32_t batch, const int32_t* draft,
                       const int32_t* target, int32_t* accept_len, int32_t* bonus,
                       int32_t* ctx_len, void* stream);

/* Same as dflash_fuse_inject, for callers that cannot set device memory
 * aside at call time -- e.g. a workspace sized with max_rows = 0 because the
 * process's device memory is owned by another allocator, or code that must
 * not grow any pool while serving.  The per-call scratch (the fused feature
 * rows, their norm statistics, the split-K partial sums and tile counters)
 * lives in one static device array compiled into the library (about 5.1 MB,
 * held by every GPU that loads the library until the process exits); the
 * caller passes only the inputs and the handle whose cache receives the
 * output.  Nothing is allocated (no cudaMalloc/cudaFree).  There is no
 * counterpart on the pages; it is a deployment variant.
 *   Limit: batch * rows_per_req <= 64 (a round's rows for up to 4 requests,
 *   or a prefill fed in chunks of 64); larger calls return
 *   DFLASH_ERR_CAPACITY and print the limit to stderr.  The two GEMMs use at
 *   most 16 CTAs, so this variant is slower than dflash_fuse_inject.
 *   The first call on a device looks up the array's device address; make
 *   that first call before any stream capture.  All calls in the process
 *   share the one array per device: calls that can overlap on the GPU (other
 *   streams, other handles on the same device) race and must be ordered by
 *   the caller.  The tile counters are cleared at the start of every call. */
DFLASH_API int dflash_fuse_inject_noalloc(dflash_handle* h, const int32_t* slots, int32_t batch, const void* feats,
                                          int32_t rows_per_req, const int32_t* n_new, void* stream);

/* Failure-detection check (no counterpart on the pages): one thread of a
 * one-warp kernel waits, through the same bounded wait the GEMM and
 * attention pipelines use, on an mbarrier that nothing ever arrives at, with
 * a limit of limit_us microseconds (1 .. 100000); it gives up, sets
 * DFLASH_DEV_TIMEOUT in the handle's status word and returns, leaving the
 * CUDA context usable.  dflash_read_status then reports (and clears) the bit.
 * The pipelines' own waits give up after 2 s the same way. */
DFLASH_API int dflash_check_wait_timeout(dflash_handle* h, uint32_t limit_us, void* stream);

/* Free a slot's pages and set its length to 0 (stream-ordered). */
DFLASH_API int dflash_reset_slot(dflash_handle* h, int32_t slot, void* stream);

/* Synchronise the device, return the device status word in *out
 * (DFLASH_DEV_* bits, 0 = clean) and clear it. */
DFLASH_API int dflash_read_status(dflash_handle* h, uint32_t* out);

DFLASH_API const char* dflash_status_string(int status);

/* ---- round graph: one CUDA graph per captured sequence of calls ---------
 * dflash_graph_begin starts capturing `stream` (thread-local mode); every
 * call enqueued on it until dflash_graph_end (library calls and the caller's
 * own kernels, e.g. the target's verify) becomes one graph, instantiated and
 * kept in the handle (replacing any previous one).  *n_kernels receives the
 * number of kernel nodes.  dflash_graph_launch replays it on `stream`. */
DFLASH_API int dflash_graph_begin(dflash_handle* h, void* stream);
DFLASH_API int dflash_graph_end(dflash_handle* h, void* stream, int32_t* n_kernels);
DFLASH_API int dflash_graph_launch(dflash_handle* h, void* stream);

/* ---- introspection ------------------------------------------------------ */

/* Copy K and V of `layer` for positions pos0..pos0+n-1 of `slot` into plain
 * [n, hkv, D] float32 DEVICE buffers (the cache itself is stored as f16,
 * pre-swizzled). */
DFLASH_API int dflash_read_kv(dflash_handle* h, int32_t layer, int32_t slot, int32_t pos0, int32_t n,
                   void* k_out, void* v_out, void* stream);

/* Current cache length of each slot in slots[batch] -> DEVICE int32 out[batch]. */
DFLASH_API int dflash_slot_lengths(dflash_handle* h, const int32_t* slots, int32_t batch, int32_t* out,
                        void* stream);

/* dflash_draft_block that also writes, when non-null, the residual stream
 * after the last layer (hidden [batch,16,H] float32) and the full logits of
 * all 16 block rows (logits [batch,16,V] float32), from the same kernels and
 * the same accumulators the argmax reads.  With block S < 16, rows S..15 of
 * each request are padding rows (finite, not part of the method). */
DFLASH_API int dflash_draft_block_debug(dflash_handle* h, const int32_t* slots, int32_t batch,
                             const int32_t* last_tok, int32_t* draft, float* hidden,
                             float* logits, void* stream);

/* ---- target model (role 1): the verify step and the trim -----------------
 * "DFlash原理深度剖析…", §三 第2步: the target runs one forward over the whole
 * block and gives, at every block position, its own next token; §三 第3步:
 * after acceptance both caches are trimmed to the confirmed length; §二.3:
 * the drafter's features are hidden states of target layers picked evenly
 * from its middle, and it shares the target's embedding and LM head.
 *
 * dflash_verify_block: block tokens [batch, 16] (DEVICE int32; row 0 the
 * last verified token, rows 1.. the drafts) at positions ctx_len ..
 * ctx_len+15 of each slot, n_valid [batch] DEVICE int32 live rows (null: 16;
 * rows >= n_valid are padding: computed, never written to the cache, never
 * keys), causal attention (row i sees the context and rows 0..i), their K/V
 * written to the slot's cache; out_tok [batch, 16] DEVICE int32 receives
 * every row's argmax (ties -> lowest id); feats, when non-null, DEVICE bf16
 * [batch, 16, n_fused, H] receives the residual stream after target layers
 * 1 + round(k (L-3) / (n_fused-1)), k = 0..n_fused-1 (the drafter's
 * dflash_fuse_inject input).  ctx_len does not move.
 * dflash_advance: ctx_len[slot] += n[b] (DEVICE int32 [batch], 0..16), the
 * positions beyond it free for the next block -- the trim after acceptance
 * (n = accept_len) and the step after a prefill chunk (n = its length).
 * Both: DFLASH_ERR_INVALID_ARG on a drafter handle or null arguments;
 * out-of-range slots and n are device-side errors (DFLASH_DEV_ARG). */
DFLASH_API int dflash_verify_block(dflash_handle* h, const int32_t* slots, int32_t batch, const int32_t* tokens,
                                   const int32_t* n_valid, int32_t* out_tok, void* feats, void* stream);
DFLASH_API int dflash_advance(dflash_handle* h, const int32_t* slots, int32_t batch, const int32_t* n,
                              void* stream);

/* dflash_verify_block at temperature T > 0: the target samples its own token
 * at every block position ("DFlash原理深度剖析…", §三 第3步: the block is
 * checked against the target's sampled tokens; "DFlash：drafter 的答案…",
 * Results: sampling at T = 1).  Row i of request b (position
 * p = ctx_len + i of slot s = slots[b]) outputs argmax_v(logit_v / T + g_v),
 * g_v = -ln(-ln u_v), u_v from the SplitMix64 stream (seed, 2, s, p) built as
 * for dflash_draft_block_sample.  Keyed by position, a position's draw is the
 * same whichever block or round it falls in, so speculative decoding with
 * dflash_accept_trim emits exactly the target's own sampled decoding (one
 * live row per call) for the same seed.  temperature < 1e-6 (or 0) is the
 * argmax; negative or NaN is DFLASH_ERR_INVALID_ARG; otherwise as
 * dflash_verify_block. */
DFLASH_API int dflash_verify_block_sample(dflash_handle* h, const int32_t* slots, int32_t batch,
                                          const int32_t* tokens, const int32_t* n_valid, float temperature,
                                          uint64_t seed, int32_t* out_tok, void* feats, void* stream);

/* a3-a6 at temperature T > 0 ([Paper walkthrough] Results and [News summary]
 * 用例与示例 report DFlash with sampling; [Code walkthrough] §三 第3步: the
 * block is checked against the target's sampled tokens with the same
 * longest-prefix rule, so dflash_accept_trim applies unchanged).  Exactly
 * dflash_draft_block, except that block row i = 1..S-1 of request b draws its
 * draft from softmax(logits / T) by the Gumbel-max rule,
 * argmax_v(logit_v / T + g_v), g_v = -ln(-ln u_v) with u_v from the
 * SplitMix64 stream (seed, 1, b, *round, i): element v is
 * mix(key + (v+1) * 0x9E3779B97F4A7C15), u = ((bits >> 41) + 0.5) * 2^-23,
 * where key folds seed then each id x as k = mix(k + 0x9E3779B97F4A7C15 * (x+1))
 * starting from mix(seed + 0x9E3779B97F4A7C15) (mix: the SplitMix64
 * finaliser).  temperature < 1e-6 (or 0) is the greedy argmax; negative or NaN
 * is DFLASH_ERR_INVALID_ARG.  round: DEVICE int32 read by the kernels (null:
 * round 0), so a captured round loop draws fresh numbers when the caller's
 * counter advances.  logits: optional DEVICE float32 [batch, 16, V]
 * receiving the unscaled logits of every block row (null: not stored). */
DFLASH_API int dflash_draft_block_sample(dflash_handle* h, const int32_t* slots, int32_t batch,
                                         const int32_t* last_tok, float temperature, uint64_t seed,
                                         const int32_t* round, int32_t* draft, float* logits, void* stream);

/* Kernel timing probe: the next n launches of kernel `kernel_id`
 * (DFLASH_KID_*) are bracketed by CUDA events recorded on the launching
 * stream (as event-record nodes when captured).  dflash_probe_read
 * synchronises on them and writes up to `cap` durations in ms. */
#define DFLASH_KID_LM_HEAD 1
#define DFLASH_KID_GATE_UP 2
#define DFLASH_KID_ATTENTION 3
#define DFLASH_KID_DOWN 4
#define DFLASH_KID_QKV 5
#define DFLASH_KID_WO 6
#define DFLASH_KID_FC 7
#define DFLASH_KID_INJECT 8
#define DFLASH_KID_ALL 255 /* dflash_trace_arm only: every GEMM and attention launch */
DFLASH_API int dflash_probe_arm(dflash_handle* h, int32_t kernel_id, int32_t n);
DFLASH_API int dflash_probe_read(dflash_handle* h, float* ms_out, int32_t cap, int32_t* n_out);

/* Timeline marks (no counterpart on the pages; measurement only).
 * dflash_marks_arm(h, n) resets the mark list and makes room for n marks;
 * each dflash_mark(h, stream) records the next mark event on `stream` (an
 * external event-record node when the stream is being captured, so a graph
 * replay records it again); marks beyond n are ignored.
 * dflash_marks_read synchronises on the recorded marks and writes up to
 * `cap` intervals in ms between consecutive marks (ms_out[i] = mark i ->
 * mark i+1); *n_out = number of intervals written. */
DFLASH_API int dflash_marks_arm(dflash_handle* h, int32_t n);
DFLASH_API int dflash_mark(dflash_handle* h, void* stream);
DFLASH_API int dflash_marks_read(dflash_handle* h, float* ms_out, int32_t cap, int32_t* n_out);

/* Device timeline of one launch: the next launch of kernel `kernel_id`
 * (DFLASH_KID_*) writes, per CTA, 8 uint64 values into the DEVICE buffer
 * buf[cap_ctas][8]; with DFLASH_KID_ALL every following GEMM and attention
 * launch takes the next rows (its grid's CTAs, in launch order) until the
 * buffer is full.  GEMMs: %globaltimer (ns) at entry, end of set-up, first
 * weight stage landed, last MMA issued, epilogue done and exit, then the
 * CTA's unit count and its SM id.  Attention (CTAs in split-fastest order):
 * entry, context length known, first page landed, pages done, partial
 * published, exit.  Launches with more CTAs than cap_ctas are not traced.
 * kernel_id 0 disarms. */
DFLASH_API int dflash_trace_arm(dflash_handle* h, int32_t kernel_id, unsigned long long* buf, int32_t cap_ctas);

/* Number of kernels this handle has launched (or captured) so far. */
DFLASH_API uint64_t dflash_launch_count(dflash_handle* h);

/* How the handle runs its kernels on this GPU, fixed at dflash_create:
 * out[0] SMs, out[1] attention splits per (request, KV head), out[2]
 * attention page loop (1 warp MMAs, 2 tcgen05), out[3] CTAs per cluster
 * sharing a GEMM token tile of 128+ tokens (1: none), out[4] how the
 * attention splits are merged (0: one thread-block cluster per request and KV
 * head, over distributed shared memory; 1: through global memory by a second
 * kernel, when that allows more splits than clusters fit at once).  out:
 * HOST int32[5].  Host only. */
DFLASH_API int dflash_plan(dflash_handle* h, int32_t* out5);

/* ---- benchmark harness: stand-in for the target's verify step -----------
 * Not part of the method.  For round r = (*round_ctr)++ it builds the
 * target tokens from the draft and caller-drawn random streams
 *   match [rounds_cap, batch, S] int32 in {0,1}, offs [rounds_cap, batch, S]
 *   int32 in [0, vocab):  t_i = d_{i+1} if match_i else offs_i (bumped to
 *   (offs_i+1) mod vocab if equal to d_{i+1}), t_{S-1} = offs_{S-1};
 * and, when feat_stream is non-null, copies the target features of the S
 * block positions ctx_len .. ctx_len+S-1 from feat_stream
 * [batch, stream_rows, n_fused*H] into feats_out [batch, S, n_fused*H]. */
/* Device timestamps of the stand-in verify (measurement only): after
 * dflash_stamps_arm(h, buf, n), the next n dflash_harness_verify calls
 * enqueued (or captured) write %globaltimer (ns) into the DEVICE buffer
 * buf[2i] when call i may start its work (the kernels before it are
 * complete) and buf[2i+1] when its last block is done.  n = 0 disarms.
 * The drafter's time in a replayed round loop is then the time outside these
 * windows, with no event-record node in the graph. */
DFLASH_API int dflash_stamps_arm(dflash_handle* h, unsigned long long* buf, int32_t n);

DFLASH_API int dflash_harness_verify(dflash_handle* h, const int32_t* slots, int32_t batch,
                          const int32_t* draft, const int32_t* match, const int32_t* offs,
                          int32_t rounds_cap, int32_t* round_ctr, int32_t* target,
                          const void* feat_stream, int32_t stream_rows, void* feats_out,
                          void* stream);

#ifdef __cplusplus
}
#endif
#endif /* DFLASH_H */
