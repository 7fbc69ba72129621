// Internal structures shared by the kernels and the host-side runtime.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dflash.h"

typedef __nv_bfloat16 bf16;
typedef __half f16;

#define DFL_MAX_LAYERS 8
#define DFL_BLOCK 16
#define DFL_PAGE 64
#ifndef DFL_BN_MAX
#define DFL_BN_MAX 256
#endif
// One packed FP8 weight block: 128 rows x 64 bytes, row-major (8 KB).
#define DFL_WBLK8_BYTES (128 * 64)
// One packed weight block: 128 rows x 64 columns of 16-bit values (16 KB).
#define DFL_WBLK_ELEMS (128 * 64)

// GEMM epilogue modes (swap-AB: weights are the 128-row A operand, tokens the N side).
enum GemmMode : int {
  GM_QKV = 0,     // layer QKV: input-norm scale, q/k head norm, RoPE; q -> q_buf, block k/v -> cache
  GM_INJECT = 1,  // fused feature -> every layer's K/V: fusion-norm scale, k norm, RoPE, paged append
  GM_RESID = 2,   // h += acc (fp32 residual); hg = f16(h * next gain); per-tile sum of squares
  GM_SWIGLU = 3,  // post-norm scale; act = silu(gate) * up (tile rows 0-63 gate, 64-127 up)
  GM_FC = 4,      // fusion projection: cg = f16(acc * fc gain); per-tile sum of squares
  GM_ARGMAX = 5   // final-norm scale; per-token argmax over the vocabulary (+ optional logits)
};

// Paged KV cache geometry (one layer's pools are at k_pool + layer*layer_stride).
struct KVGeom {
  f16* k_pool;
  f16* v_pool;
  long long layer_stride;  // elements between layers' pools
  const int* page_table;   // [max_slots][max_pages_per_slot]
  int max_pages_per_slot;
  int max_pages;
  int hkv, D;
};

struct GemmParams {
  // problem
  int M;            // token rows of B
  int N;            // output rows (features) per group
  int kblocks;      // K / 64
  int n_tiles;      // tiles per group along N
  int t_tiles;      // token tiles
  int BN;           // token tile (multiple of 16, <= 256)
  int groups;       // A operands used (grouped inject: one per layer)
  int total_tiles;  // groups * n_tiles * t_tiles
  int cl;           // CTAs per cluster sharing each token tile (1, or 4 for token tiles >= 128)
  int n_tg;         // n-tile groups of cl per group: ceil(n_tiles / cl)
  int total_ctiles; // scheduled tiles: groups * n_tg * t_tiles (the cluster's ranks take the cl n-tiles)
  int allow_split;  // 0: every tile in one CTA over the full K
  int stages;
  int red_items;    // split-K part chunks (8 KB) the reduction buffer holds (gemm_red_items)
  int tmem_cols;    // power of two >= max(32, 2*BN)
  uint32_t ab_type; // 0: f16 operands, 1: bf16 operands
  const void* a[DFL_MAX_LAYERS];  // packed A blocks [tiles][kblocks][128x64] per group
  int a_fp8;                      // 1: A blocks are FP8 E4M3 (8 KB, row-major), converted to f16 in the SM
  const float* a_scale[DFL_MAX_LAYERS];  // a_fp8: per packed row scale [tiles * 128] per group
  int a_tile_off;   // first packed tile of the range (inject: hq*D/128)
  int mode;
  const int* m_dyn;     // non-null: the launch computes the first *m_dyn (<= M) token rows (device count)
  const int* row_map;   // INJECT over compacted rows: row j's source row b * rows_per_req + i
  // shapes for epilogues
  int H;            // hidden (norm width for ss partial consumers)
  int hq, hkv, D;
  int rows_per_req; // inject: feature rows per request; QKV/ARGMAX: block (16)
  float eps;
  // norm scales
  const float* ss_in;  // [ss_parts][ss_ld] sums of squares of the normalised input
  int ss_parts;
  int ss_ld;           // leading dimension of ss_in (token rows of the producer)
  // QKV with folded KV injection: token rows >= inj_m0 are fused-feature rows
  // (request (t-inj_m0)/rows_per_req), scaled by ss_inj [ss_parts][inj_ld]
  int inj_m0;          // 0: no injection rows
  const float* ss_inj;
  int inj_ld;
  float* ss_out;       // [n_tiles][M]
  // tensors
  float* h;             // RESID: fp32 residual [M][N]
  f16* out;             // QKV: q_buf [M][hq*D]; RESID: hg [M][N]; SWIGLU: act [M][I]; FC: cg [M][N]
  const float* gain;    // RESID: next norm gain; FC: fusion gain
  const float* qn_gain; // QKV: q head-norm gain [D]
  const float* kn_gain[DFL_MAX_LAYERS];  // per group (inject) / [0] (QKV)
  int layer;            // QKV: layer index for the cache
  KVGeom kv;
  const int* slots;     // [batch]
  const int* ctx_len;   // [max_slots] (QKV: block starts here)
  const int* pos0;      // [batch] (inject: request b's first new position)
  const int* n_eff;     // [batch] (inject: rows appended)
  const float2* rope;   // [max_pos][D/2] (cos, sin)
  int max_pos;
  const int2* bctx;     // QKV: block tokens' {position, page} (BlockCtx)
  const float2* brope;  // QKV: block tokens' RoPE rows [M][D/2]
  // argmax
  unsigned long long* keys;  // [M]
  float* logits;             // optional [M][N] (N = vocab)
  int* draft;                // [batch][block-1]
  int block;                 // ARGMAX: block size S (drafts from rows 1..S-1); 16 rows per request either way
  int row0;                  // ARGMAX: first block row whose token is output (1: drafts; 0: target verify)
  float temp_inv;            // ARGMAX: 1/temperature (0: greedy argmax)
  unsigned long long seed;   // ARGMAX sampling: stream seed
  const int* round;          // ARGMAX sampling: round index (device; null: 0)
  unsigned* done_ctr;
  // optional timeline: [grid][8] %globaltimer stamps per CTA (null: off)
  unsigned long long* trace;
  // split-K scratch
  float* ws;            // [grid][2][BN_MAX*128]
  unsigned* tile_ctr;   // [total_tiles] parts arrived (self-resetting)
  unsigned* tile_fin;   // [total_tiles] finalisers done, when several share a tile (self-resetting)
  uint32_t* status;
};

struct AttnParams {
  const f16* q;     // [M][hq][D]
  f16* out;         // [M][hq][D]
  KVGeom kv;
  int layer;
  const int* slots;
  const int* ctx_len;  // keys = ctx_len + block (block K/V already in the cache)
  int hq, hkv, D;
  int n_splits;        // CTAs per (request, KV head): one cluster (<= 16), or any count with merge_global
  int merge_global;    // 1: splits write partials to `part`, k_attn_merge combines them (no cluster)
  float* part;         // [batch * hkv][n_splits][attn_part_floats(D)] partials (merge_global)
  int block;           // block size S: keys = context + S (rows S..15 of a request are padding)
  int causal;          // target verify: block row t sees keys < ctx + min(t, n_valid-1) + 1
  int early;           // 1: the page list and the pages holding no block row are read before the wait on
                       // the QKV projection (which then wrote no context row: not a folded injection)
  const int* n_valid;  // causal: [batch] live rows (null: block); keys = context + n_valid
  const int* order;    // [batch] request of grid row z (null: z itself): longest first, so the CTAs of
                       // the longest requests start first and the short ones fill the last wave
  float scale_log2;    // log2(e) / sqrt(D)
  uint32_t* status;
  unsigned long long* trace;  // optional [grid][8] timeline (null: off)
};

// host launchers (gemm.cu / attention.cu / small.cu)
size_t gemm_smem_bytes(int BN, int stages, int fp8);
int gemm_red_items(int BN, int stages, int fp8);
int gemm_pick_stages(int BN, int mode, int fp8);
cudaError_t gemm_launch(const CUtensorMap& B, const GemmParams& p, int grid, cudaStream_t s, bool pdl);
// Clusters of `cl` GEMM CTAs (token tile BN, `stages` ring) the GPU holds at once.
int gemm_max_clusters(int BN, int stages, int cl);
cudaError_t gemm_init_attributes();

// Floats of one split's partial: [128 rows][D + 4] unnormalised O, then the
// rows' running maxima and sums.
constexpr int attn_part_floats(int D) { return 128 * (D + 4) + 2 * 128; }

// Attention clusters of `splits` CTAs the GPU can hold at once (0: cannot
// launch); tc selects the tcgen05 page loop, else the warp-MMA one.
int attn_max_active_clusters(int D, int hq, int hkv, int splits, bool tc);
cudaError_t attn_launch(const AttnParams& p, int batch, cudaStream_t s, bool pdl, bool tc);
cudaError_t attn_init_attributes();

// weight preparation (dflash_create)
cudaError_t launch_pack_weight(const bf16* src, void* dst, int N, int K, int n_tiles, int swiglu_I, bool to_f16,
                               uint32_t* status, cudaStream_t s);
cudaError_t launch_gain_f32(const bf16* src, float* dst, int n, cudaStream_t s);
// FP8 E4M3 packing with per-row scales (packed row order): scale = max|row| / 448,
// q = E4M3(w / scale) rounded to nearest even, saturating.
cudaError_t launch_pack_weight_fp8(const bf16* src, uint8_t* dst, float* scale, int N, int K, int n_tiles,
                                   int swiglu_I, cudaStream_t s);

// Positions, pages and RoPE rows of a round's block tokens: the same for
// every layer, so the embedding kernel writes them once for the layers' QKV
// epilogues (bctx[t] = {position, page or -1}, brope[t][D/2] = (cos, sin)).
struct BlockCtx {
  const int* ctx_len;
  const int* page_table;
  int max_pages_per_slot, max_pages;
  const float2* rope;
  int D, max_pos;
  int block;  // block size S (rows S..15 of each request are padding)
  const int* tokens;   // target verify: [batch][16] block tokens (null: last_tok + masks)
  const int* n_valid;  // target verify: [batch] live rows (null: block)
  int max_slots;
  int* slots_ok;  // [batch] out: slots with out-of-range ones replaced by 0
  int2* bctx;
  float2* brope;
  int* order;  // [batch] out (null: not written): the requests by descending key count, for the attention grid
};
cudaError_t launch_embed(const int* slots, int batch, const int* last_tok, int mask_id, int vocab,
                         const void* embed_pk, const float* embed_scale, const float* gain, int H, float* h, f16* hg,
                         float* ss,
                         unsigned long long* keys, const BlockCtx& bc, uint32_t* status, cudaStream_t s);
cudaError_t launch_page_alloc(const int* slots, int batch, int S, const int* n_new, int rows_per_req, int* ctx_len,
                              int* pos0, int* n_pages, int* page_table, int max_pages_per_slot,
                              int* free_stack, int* free_top, int* n_eff, int* slots_ok, int max_slots,
                              uint32_t* status, cudaStream_t s, int* row_off = nullptr, int* n_live = nullptr);
// The appended feature rows of a round gathered densely: request b's first
// n_eff[b] rows of feats [batch][rows_per_req][F] to rows row_off[b].. of
// dst [*, F], row_map[j] = source row of dst row j.
cudaError_t launch_compact_rows(const bf16* feats, int batch, int rows_per_req, int F, const int* n_eff,
                                const int* row_off, bf16* dst, int* row_map, cudaStream_t s);
cudaError_t launch_accept(const int* slots, int batch, int S, const int* draft, const int* target, int* accept_len,
                          int* bonus, int* ctx_out, int* ctx_len, int max_slots, uint32_t* status,
                          cudaStream_t s);
cudaError_t launch_reset_slot(int slot, int* ctx_len, int* n_pages, int* page_table,
                              int max_pages_per_slot, int* free_stack, int* free_top, cudaStream_t s);
cudaError_t launch_pool_init(int* free_stack, int* free_top, int max_pages, cudaStream_t s);
cudaError_t launch_rope_table(float2* tab, int max_pos, int D, float theta, cudaStream_t s);
cudaError_t launch_read_kv(const KVGeom& kv, int layer, int slot, int pos0, int n, float* k_out, float* v_out,
                           cudaStream_t s);
cudaError_t launch_slot_lengths(const int* slots, int batch, const int* ctx_len, int max_slots, int* out,
                                cudaStream_t s);
// Rows of the residual stream h [M][H] (fp32) into feats [M][n_fused][H]
// (bf16) at index `tap` (the target's fused-feature outputs).
cudaError_t launch_wait_check(uint32_t* status, unsigned long long limit_ns, cudaStream_t s);
cudaError_t launch_tap(const float* h, int M, int H, bf16* feats, int tap, int n_fused, cudaStream_t s);
cudaError_t launch_harness_verify(const int* slots, int batch, int S, const int* draft, const int* match,
                                  const int* offs, int rounds_cap, int* round_ctr, int* target, int vocab,
                                  const bf16* feat_stream, int stream_rows, bf16* feats_out, int F,
                                  const int* ctx_len, int max_slots, unsigned long long* stamp,
                                  unsigned* blocks_done, cudaStream_t s);
