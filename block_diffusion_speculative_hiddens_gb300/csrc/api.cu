// Host runtime behind the C ABI of include/dflash.h: configuration checks,
// workspace layout, TMA descriptors, launch planning, CUDA-graph capture and
// kernel timing probes.  Every entry point returns a dflash_status; nothing
// throws across the boundary and nothing here allocates device memory (the
// caller supplies the workspace).
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "common.cuh"
#include "internal.h"

namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool load_encode() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

// 2-D 16-bit tensor [rows, cols] row-major (f16 or bf16); box = 64 columns
// (128 B) x box_rows, 128-byte swizzle -- the canonical K-major tcgen05
// operand layout.
bool make_tmap(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
               bool is_bf16 = false) {
  if (!load_encode()) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = g_encode(m, is_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct Carve {
  size_t off = 0;
  char* base = nullptr;
  template <class T>
  T* take(size_t n) {
    off = align_up(off, 256);
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off += n * sizeof(T);
    return p;
  }
};

int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }

struct Probe {
  int kid = 0;
  int n = 0;
  int next = 0;
  std::vector<cudaEvent_t> ev;  // 2*n
};

struct Trace {
  int kid = 0;  // DFLASH_KID_*, or DFLASH_KID_ALL: every GEMM and attention launch in turn
  unsigned long long* buf = nullptr;
  int cap = 0;  // CTAs the buffer holds
  int used = 0; // DFLASH_KID_ALL: rows taken by the launches so far
  // Rows of buf for the next launch of kernel `kid` (null: not traced).
  unsigned long long* take(int k, long long ctas) {
    if (!buf || !k) return nullptr;
    if (kid == DFLASH_KID_ALL) {
      if (used + ctas > cap) return nullptr;
      unsigned long long* r = buf + (size_t)used * 8;
      used += (int)ctas;
      return r;
    }
    if (kid != k || ctas > cap) return nullptr;
    kid = 0;  // one launch only
    return buf;
  }
};

}  // namespace

struct dflash_handle {
  dflash_config cfg;
  int num_sms = 0;
  int gemm_cl = 1;       // CTAs per cluster sharing a token tile of 128+ tokens
  int gemm_cl_ctas = 0;  // CTAs of such clusters the GPU holds at once
  int max_tok = 0;     // max_batch * block
  int max_pos = 0;     // max_pages_per_slot * page_size
  int attn_splits = 1;
  bool attn_tc = false;      // tcgen05 attention page loop
  bool attn_global = false;  // splits merged through global memory (no cluster)
  float* attn_part = nullptr;
  int* attn_order = nullptr;  // [max_batch] the attention grid's request order (longest first)
  int max_tiles = 0;
  // weights, copied into the workspace at create: matrices packed into
  // 128x64 blocks (f16, except the bf16 fusion projection), gains as fp32
  f16* embed_pk;
  bf16* fc_pk;
  f16* wqkv_pk[DFL_MAX_LAYERS];
  f16* wo_pk[DFL_MAX_LAYERS];
  f16* gu_pk[DFL_MAX_LAYERS];
  f16* down_pk[DFL_MAX_LAYERS];
  // FP8 weights: the packed blocks above hold E4M3 bytes; per packed row scales
  bool fp8 = false;
  float* embed_sc = nullptr;
  float *wqkv_sc[DFL_MAX_LAYERS] = {}, *wo_sc[DFL_MAX_LAYERS] = {}, *gu_sc[DFL_MAX_LAYERS] = {},
        *down_sc[DFL_MAX_LAYERS] = {};
  float* fc_norm;
  float* final_norm;
  float* in_norm[DFL_MAX_LAYERS];
  float* q_norm[DFL_MAX_LAYERS];
  float* k_norm[DFL_MAX_LAYERS];
  float* post_norm[DFL_MAX_LAYERS];
  // cached B operand descriptors for the current token count
  int bm_M = -1;
  CUtensorMap tm_hg, tm_o, tm_act;
  CUtensorMap tm_hg_s;  // hg in DFL_BN_SMALL-row token tiles (the QKV projection)
  int bm_MX = -1;
  CUtensorMap tm_hgx;  // hg plus the fused-feature rows below it
  int bm_rows = -1;
  CUtensorMap tm_cg;
  // round injections of more rows than one token tile: the appended rows
  // gathered densely (compact), their source rows and count
  bf16* cstage = nullptr;  // [max_batch * 16][n_fused * H]
  int* row_map = nullptr;  // [max_batch * 16]
  int* row_off = nullptr;  // [max_batch]
  int* n_live = nullptr;   // [1]
  int bm_cstage = -1;
  CUtensorMap tm_cstage;
  // workspace
  uint32_t* status;
  int *ctx_len, *pos0, *n_pages, *page_table, *free_stack, *free_top, *n_eff;
  int* slots_ok;  // [max_batch] the call's slots, out-of-range ones replaced by 0 (read by GEMMs, attention)
  f16 *k_pool, *v_pool;
  long long layer_stride;
  float2* rope;
  float* h;
  f16 *hg, *qbuf, *obuf, *act, *cg;
  float *ss_a, *ss_c;
  unsigned long long* keys;
  int2* bctx;
  float2* brope;
  unsigned* done_ctr;
  float* gemm_ws;
  unsigned* tile_ctr;
  // runtime
  bool pdl = true;
  uint64_t launches = 0;
  Probe probe;
  Probe marks;  // timeline marks: ev[i] = mark i, n = capacity, next = recorded
  Trace trace;
  unsigned long long* stamps = nullptr;  // harness verify stamps [stamp_cap][2] (null: off)
  int stamp_cap = 0, stamp_next = 0;
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
};

namespace {

bool cfg_valid(const dflash_config* c) {
  if (!c) return false;
  if (c->hidden <= 0 || c->n_q_heads <= 0 || c->n_kv_heads <= 0 || c->head_dim <= 0 || c->intermediate <= 0 ||
      c->n_layers <= 0 || c->vocab <= 0 || c->n_fused <= 0)
    return false;
  if (c->n_layers > DFL_MAX_LAYERS) return false;
  // block: the trained size is 16; inference may use a smaller block S (rows
  // S..15 of a request are carried as padding and never become keys)
  if (c->block < 2 || c->block > DFL_BLOCK || c->page_size != DFL_PAGE) return false;
  if (c->head_dim != 64 && c->head_dim != 128) return false;
  if (c->hidden % 128 || c->hidden > 8192) return false;
  if (c->intermediate % 64) return false;
  if ((c->n_q_heads * c->head_dim) % 128 || (c->n_kv_heads * c->head_dim) % 128) return false;
  if (c->n_q_heads % c->n_kv_heads) return false;
  const int G = c->n_q_heads / c->n_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8) return false;
  if (c->max_batch <= 0 || c->max_batch > 64 || c->max_slots <= 0 || c->max_pages <= 0 ||
      c->max_pages_per_slot <= 0 || c->max_rows < 0)
    return false;
  if (c->mask_id < 0 || c->mask_id >= c->vocab) return false;
  if (!(c->rms_eps > 0.f) || !(c->rope_theta > 1.f)) return false;
  if (c->attn_impl < 0 || c->attn_impl > 2) return false;
  if (c->role != 0 && c->role != 1) return false;
  if (c->weight_fp8 != 0 && c->weight_fp8 != 1) return false;
  // a target: full 16-token blocks, and 5 distinct middle layers to tap
  if (c->role == 1 && (c->block != DFL_BLOCK || c->n_layers < c->n_fused + 2)) return false;
  return true;
}

// Target layers whose outputs are the drafter's features, shallow to deep:
// layers 1..L-2 evenly spread (round half up of k(L-3)/(n-1)).
int tap_layer(int k, int L, int n) { return 1 + (2 * k * (L - 3) + (n - 1)) / (2 * (n - 1)); }

#ifndef DFL_ATTN_MAX_SPLITS
#define DFL_ATTN_MAX_SPLITS 16
#endif

// Split-KV count: about one wave of CTAs, at least 4 pages per split at full
// slot capacity, at most 16 (one thread-block cluster).  dflash_create then
// lowers it until the GPU can hold a cluster for every (request, KV head) at
// once (clusters are placed within one GPC each).
int pick_attn_splits(const dflash_config& c, int num_sms) {
  const int pairs = c.max_batch * c.n_kv_heads;
  int want = ceil_div(num_sms, pairs);
  want = std::min(want, std::max(1, c.max_pages_per_slot / 4));
  want = std::min(want, DFL_ATTN_MAX_SPLITS);
  return std::max(1, want);
}

// Split-KV count without a cluster: every CTA of one launch resident at once
// (one per SM), at least 4 pages per split at full slot capacity, at most 32;
// the splits' partials are then merged by a second kernel.
#ifndef DFL_ATTN_GLOBAL
#define DFL_ATTN_GLOBAL 1
#endif
// Token tiles of at most DFL_BN_SMALL rows for the GEMMs with few n-tiles
// and heavy epilogues (QKV, fusion, injection) over at most
// DFL_BN_SMALL_ROWS rows: at a round's 1,024 rows twice the token tiles give
// their CTAs whole tiles instead of shares of a few split ones (measured on
// GB300, batched round 4,411 -> 4,313 us: QKV 534 -> 487 us, injection 128
// -> 80 us; the lm_head and gate/up lose with it, their tiles being
// plentiful, and so does a 2,048-row prefill chunk: 44.2 -> 48.0 ms).
#ifndef DFL_BN_SMALL
#define DFL_BN_SMALL 128
#endif
#ifndef DFL_BN_SMALL_ROWS
#define DFL_BN_SMALL_ROWS 1024
#endif
int bn_small(int M) { return M <= DFL_BN_SMALL_ROWS ? DFL_BN_SMALL : DFL_BN_MAX; }

#ifndef DFL_ATTN_GLOBAL_MIN_PAGES  // pages per split (at full slot capacity) from which splits merge through memory
#define DFL_ATTN_GLOBAL_MIN_PAGES 32
#endif
#ifndef DFL_ATTN_BATCH_SPLITS  // splits per (request, KV head) when the pairs alone fill the SMs
#define DFL_ATTN_BATCH_SPLITS 1
#endif
int global_attn_splits(const dflash_config& c, int num_sms) {
  const int pairs = c.max_batch * c.n_kv_heads;
  int want = pairs >= num_sms ? DFL_ATTN_BATCH_SPLITS : num_sms / pairs;
  want = std::min(want, std::max(1, c.max_pages_per_slot / 4));
  return std::max(1, std::min(want, 32));
}

// Lay out the workspace; with base == nullptr only sizes are computed.
size_t carve(dflash_handle* h, const dflash_config& c, char* base, int num_sms) {
  Carve w;
  w.base = base;
  const int M = c.max_batch * DFL_BLOCK;
  const int R = std::max(c.max_rows, 1);
  const int H = c.hidden, D = c.head_dim, hq = c.n_q_heads, hkv = c.n_kv_heads, I = c.intermediate;
  const int max_pos = c.max_pages_per_slot * DFL_PAGE;
  const long long blk = 64LL * hkv * D;  // elements per page per layer (K or V)
  const long long layer_stride = (long long)c.max_pages * blk;
  const int splits = pick_attn_splits(c, num_sms);
  // split-K tile counters: the largest tile count of any GEMM (all of them,
  // the lm_head included, use the balanced split)
  const int t_tiles_max = ceil_div(std::max(M, R), DFL_BN_MAX);
  int tiles = std::max({(c.n_q_heads + 2 * hkv) * D / 128, H / 128, I / 64, c.n_layers * 2 * hkv * D / 128,
                        ceil_div(c.vocab, 128)});
  tiles *= t_tiles_max;
  // the GEMMs on DFL_BN_SMALL-row token tiles: QKV, fusion, injection
  tiles = std::max(tiles, std::max({(c.n_q_heads + 2 * hkv) * D / 128, H / 128, c.n_layers * 2 * hkv * D / 128}) *
                              ceil_div(std::min(std::max(M, R), DFL_BN_SMALL_ROWS), DFL_BN_SMALL));

  dflash_handle tmp;
  dflash_handle* o = h ? h : &tmp;
  o->status = w.take<uint32_t>(64);
  o->ctx_len = w.take<int>(c.max_slots);
  o->pos0 = w.take<int>(c.max_batch);
  o->n_pages = w.take<int>(c.max_slots);
  o->page_table = w.take<int>((size_t)c.max_slots * c.max_pages_per_slot);
  o->free_stack = w.take<int>(c.max_pages);
  o->free_top = w.take<int>(1);
  o->n_eff = w.take<int>(c.max_batch);
  o->slots_ok = w.take<int>(c.max_batch);
  const size_t KBh = H / 64;
  // packed blocks: 16 KB of f16, or 8 KB of FP8 (+ a float scale per packed row)
  const bool f8 = c.weight_fp8 != 0;
  auto blocks = [&](size_t n_blk) {
    return reinterpret_cast<f16*>(w.take<uint8_t>(n_blk * (f8 ? DFL_WBLK8_BYTES : DFL_WBLK_ELEMS * 2)));
  };
  auto scales = [&](size_t n_tiles) { return f8 ? w.take<float>(n_tiles * 128) : nullptr; };
  o->embed_pk = blocks((size_t)ceil_div(c.vocab, 128) * KBh);
  o->embed_sc = scales((size_t)ceil_div(c.vocab, 128));
  o->fc_pk = w.take<bf16>((size_t)(H / 128) * (c.n_fused * H / 64) * DFL_WBLK_ELEMS);
  o->fc_norm = w.take<float>(H);
  o->final_norm = w.take<float>(H);
  for (int l = 0; l < c.n_layers; ++l) {
    o->wqkv_pk[l] = blocks((size_t)((hq + 2 * hkv) * D / 128) * KBh);
    o->wo_pk[l] = blocks((size_t)(H / 128) * (hq * D / 64));
    o->gu_pk[l] = blocks((size_t)(I / 64) * KBh);
    o->down_pk[l] = blocks((size_t)(H / 128) * (I / 64));
    o->wqkv_sc[l] = scales((size_t)((hq + 2 * hkv) * D / 128));
    o->wo_sc[l] = scales((size_t)(H / 128));
    o->gu_sc[l] = scales((size_t)(I / 64));
    o->down_sc[l] = scales((size_t)(H / 128));
    o->in_norm[l] = w.take<float>(H);
    o->post_norm[l] = w.take<float>(H);
    o->q_norm[l] = w.take<float>(D);
    o->k_norm[l] = w.take<float>(D);
  }
  o->k_pool = w.take<f16>((size_t)c.n_layers * layer_stride);
  o->v_pool = w.take<f16>((size_t)c.n_layers * layer_stride);
  o->layer_stride = layer_stride;
  o->rope = w.take<float2>((size_t)max_pos * (D / 2));
  o->h = w.take<float>((size_t)M * H);
  o->hg = w.take<f16>((size_t)2 * M * H);  // [block rows ; fused-feature rows of a folded round]
  o->ss_a = w.take<float>((size_t)(H / 128) * M);
  o->qbuf = w.take<f16>((size_t)M * hq * D);
  o->obuf = w.take<f16>((size_t)M * hq * D);
  o->act = w.take<f16>((size_t)M * I);
  o->keys = w.take<unsigned long long>(M);
  o->bctx = w.take<int2>(M);
  o->attn_order = w.take<int>(c.max_batch);
  o->brope = w.take<float2>((size_t)M * (D / 2));
  o->done_ctr = w.take<unsigned>(64);
  o->cg = w.take<f16>((size_t)R * H);
  o->ss_c = w.take<float>((size_t)(H / 128) * R);
  o->gemm_ws = w.take<float>((size_t)num_sms * 2 * DFL_BN_MAX * 128);
  {
    const int gs = DFL_ATTN_GLOBAL ? global_attn_splits(c, num_sms) : 1;
    o->attn_part = gs > 1 ? w.take<float>((size_t)c.max_batch * hkv * gs * attn_part_floats(D)) : nullptr;
  }
  o->tile_ctr = w.take<unsigned>(2 * (size_t)tiles);  // arrivals, then finalisers done
  if (M > DFL_BN_MAX && c.role == 0) {  // a round's injection can span several token tiles: compaction buffers
    o->cstage = w.take<bf16>((size_t)M * c.n_fused * H);
    o->row_map = w.take<int>(M);
    o->row_off = w.take<int>(c.max_batch);
    o->n_live = w.take<int>(1);
  } else {
    o->cstage = nullptr;
    o->row_map = o->row_off = o->n_live = nullptr;
  }
  if (h) {
    h->attn_splits = splits;
    h->max_tiles = tiles;
    h->max_pos = max_pos;
    h->max_tok = M;
  }
  return align_up(w.off, 256);
}

int device_sms(int dev) {
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

inline int cuda_err(cudaError_t e) {
  if (e == cudaSuccess) return DFLASH_OK;
  fprintf(stderr, "[dflash] CUDA error: %s\n", cudaGetErrorString(e));
  return DFLASH_ERR_CUDA;
}

// Event pair around one launch: event-record nodes when the stream is being
// captured, plain records otherwise.
struct ProbeScope {
  dflash_handle* h;
  cudaStream_t s;
  bool on = false;
  bool capturing = false;
  int idx = 0;
  void record(cudaEvent_t e) {
    if (capturing)
      cudaEventRecordWithFlags(e, s, cudaEventRecordExternal);
    else
      cudaEventRecord(e, s);
  }
  ProbeScope(dflash_handle* h_, int kid, cudaStream_t s_) : h(h_), s(s_) {
    if (kid && h->probe.kid == kid && h->probe.next < h->probe.n) {
      on = true;
      idx = h->probe.next++;
      cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
      capturing = cudaStreamIsCapturing(s, &st) == cudaSuccess && st == cudaStreamCaptureStatusActive;
      record(h->probe.ev[2 * idx]);
    }
  }
  ~ProbeScope() {
    if (on) record(h->probe.ev[2 * idx + 1]);
  }
};

#ifndef DFL_GEMM_MAX_CL
#define DFL_GEMM_MAX_CL 4
#endif

// Token tiling of an M-row GEMM operand: t_tiles tiles of BN <= bn_max rows;
// for tiles of 128 tokens or more, cl CTAs of a cluster share each token
// tile (each loads BN/cl rows into all of them), so its box is BN/cl rows.
struct GemmShape {
  int t_tiles, BN, cl;
  uint32_t box() const { return (uint32_t)(BN / cl); }
};
GemmShape gemm_shape(const dflash_handle* h, int M, int bn_max = DFL_BN_MAX) {
  GemmShape g;
  g.t_tiles = ceil_div(std::max(M, 1), bn_max);
  g.BN = ((ceil_div(std::max(M, 1), g.t_tiles) + 15) / 16) * 16;
  g.cl = (g.BN >= 128 && h->gemm_cl > 1) ? h->gemm_cl : 1;
  if (g.cl == 4) g.BN = (g.BN + 31) / 32 * 32;  // each quarter whole 8-row swizzle atoms
  return g;
}

// FP8 weights: the GEMM streams E4M3 blocks and scales rows by `sc` (group g)
void fp8_weights(const dflash_handle* h, GemmParams& p, const float* sc, int g = 0) {
  if (!h->fp8) return;
  p.a_fp8 = 1;
  p.a_scale[g] = sc;
}

// Plan and launch one GEMM over packed A operands a[0..groups-1] (tiles
// a_tile_off .. a_tile_off+n_tiles-1 of each) and the token operand B.
int run_gemm(dflash_handle* h, cudaStream_t s, int mode, const void* const* a, int groups, int a_tile_off,
             int n_tiles, int K, const CUtensorMap& B, int M, GemmParams p, bool allow_split, uint32_t ab_type,
             int kid = 0, int bn_max = DFL_BN_MAX) {
  if (M <= 0) return DFLASH_OK;
  const GemmShape gs = gemm_shape(h, M, bn_max);
  const int t_tiles = gs.t_tiles;
  const int BN = gs.BN;
  p.mode = mode;
  p.M = M;
  if (!p.ss_ld) p.ss_ld = M;
  p.kblocks = K / 64;
  p.n_tiles = n_tiles;
  p.t_tiles = t_tiles;
  p.BN = BN;
  p.groups = groups;
  for (int g = 0; g < groups; ++g) p.a[g] = a[g];
  p.a_tile_off = a_tile_off;
  p.ab_type = ab_type;
  p.total_tiles = groups * n_tiles * t_tiles;
  p.cl = gs.cl;
  p.n_tg = ceil_div(n_tiles, gs.cl);
  p.total_ctiles = groups * p.n_tg * t_tiles;
  p.allow_split = allow_split ? 1 : 0;
  p.stages = gemm_pick_stages(BN, mode, p.a_fp8);
  p.red_items = gemm_red_items(BN, p.stages, p.a_fp8);
  int cols = 32;
  while (cols < 2 * BN) cols *= 2;
  p.tmem_cols = cols;
  p.status = h->status;
  p.ws = h->gemm_ws;
  p.tile_ctr = h->tile_ctr;
  p.tile_fin = h->tile_ctr + h->max_tiles;
  p.eps = h->cfg.rms_eps;
  p.H = h->cfg.hidden;
  p.hq = h->cfg.n_q_heads;
  p.hkv = h->cfg.n_kv_heads;
  p.D = h->cfg.head_dim;
  p.rope = h->rope;
  p.max_pos = h->max_pos;
  if (allow_split && p.total_tiles > h->max_tiles) return DFLASH_ERR_SHAPE;
  const long long units = allow_split ? (long long)p.total_ctiles * p.kblocks : p.total_ctiles;
  const int clusters = (int)std::min<long long>(units, gs.cl > 1 ? h->gemm_cl_ctas / gs.cl : h->num_sms);
  const int grid = clusters * gs.cl;
  if (units * (clusters + 1) >= (1LL << 31)) return DFLASH_ERR_SHAPE;  // the kernel's unit math is 32-bit
  if (unsigned long long* tb = h->trace.take(kid, grid)) p.trace = tb;
  ProbeScope ps(h, kid, s);
  h->launches++;
  return cuda_err(gemm_launch(B, p, grid, s, h->pdl));
}

KVGeom kv_geom(dflash_handle* h) {
  KVGeom g;
  g.k_pool = h->k_pool;
  g.v_pool = h->v_pool;
  g.layer_stride = h->layer_stride;
  g.page_table = h->page_table;
  g.max_pages_per_slot = h->cfg.max_pages_per_slot;
  g.max_pages = h->cfg.max_pages;
  g.hkv = h->cfg.n_kv_heads;
  g.D = h->cfg.head_dim;
  return g;
}

int ensure_bmaps(dflash_handle* h, int M) {
  if (h->bm_M == M) return DFLASH_OK;
  const dflash_config& c = h->cfg;
  const uint32_t BN = gemm_shape(h, M).box();
  if (!make_tmap(&h->tm_hg, h->hg, M, c.hidden, BN)) return DFLASH_ERR_CUDA;
  if (!make_tmap(&h->tm_hg_s, h->hg, M, c.hidden, gemm_shape(h, M, bn_small(M)).box())) return DFLASH_ERR_CUDA;
  if (!make_tmap(&h->tm_o, h->obuf, M, (uint64_t)c.n_q_heads * c.head_dim, BN)) return DFLASH_ERR_CUDA;
  if (!make_tmap(&h->tm_act, h->act, M, c.intermediate, BN)) return DFLASH_ERR_CUDA;
  h->bm_M = M;
  return DFLASH_OK;
}

// Draft one block; with `feats` non-null, first fuse the new feature rows and
// fold their K/V injection into every layer's QKV projection (rows M.. of its
// token operand), so each layer's K/V weights stream once per round.
struct Sampling {
  float temp_inv = 0.f;  // 0: greedy
  unsigned long long seed = 0;
  const int32_t* round = nullptr;
};

// A target model's verify pass: the block's real tokens, its live rows,
// the fused-feature taps and every row's token.
struct Verify {
  const int32_t* tokens = nullptr;   // [batch][16]
  const int32_t* n_valid = nullptr;  // [batch] (null: 16)
  bf16* feats = nullptr;             // [batch][16][n_fused][H] (null: not written)
};

int draft_impl(dflash_handle* h, const int32_t* slots, int32_t batch, const int32_t* last_tok, int32_t* draft,
               float* hidden, float* logits, void* stream, const void* feats = nullptr, int rows_per_req = 0,
               const int32_t* n_new = nullptr, Sampling smp = Sampling(), Verify vf = Verify()) {
  if (!h || batch < 0 || batch > h->cfg.max_batch) return DFLASH_ERR_INVALID_ARG;
  if (batch == 0) return DFLASH_OK;
  const bool target = vf.tokens != nullptr;
  if (!slots || (!last_tok && !target) || !draft) return DFLASH_ERR_INVALID_ARG;
  if (cudaSetDevice(h->cfg.device) != cudaSuccess) return DFLASH_ERR_CUDA;
  cudaStream_t s = (cudaStream_t)stream;
  const dflash_config& c = h->cfg;
  const int M = batch * DFL_BLOCK;
  const int H = c.hidden, D = c.head_dim, hq = c.n_q_heads, hkv = c.n_kv_heads, I = c.intermediate;
  int rc = ensure_bmaps(h, M);
  if (rc) return rc;
  const KVGeom kv = kv_geom(h);
  const bool fold = feats != nullptr;
  const int R = fold ? batch * rows_per_req : 0;
  CUtensorMap tm_feats;
  if (fold) {
    // every descriptor is encoded (and the caller's feature rows checked)
    // before anything is queued, so a refused call leaves the slots untouched
    const int MX = M + R;
    if (!make_tmap(&tm_feats, feats, R, (uint64_t)c.n_fused * H, gemm_shape(h, R).box(), true))
      return DFLASH_ERR_INVALID_ARG;
    if (h->bm_MX != MX) {
      if (!make_tmap(&h->tm_hgx, h->hg, MX, H, gemm_shape(h, MX).box())) return DFLASH_ERR_CUDA;
      h->bm_MX = MX;
    }
    h->launches++;
    rc = cuda_err(launch_page_alloc(slots, batch, h->cfg.block, n_new, rows_per_req, h->ctx_len, h->pos0, h->n_pages,
                                    h->page_table, c.max_pages_per_slot, h->free_stack, h->free_top, h->n_eff, h->slots_ok,
                                    c.max_slots, h->status, s));
    if (rc) return rc;
    GemmParams p = {};
    p.out = h->hg + (size_t)M * H;  // fused-feature rows right below the block rows
    p.gain = h->fc_norm;
    p.ss_out = h->ss_c;
    p.N = H;
    const void* a = h->fc_pk;
    rc = run_gemm(h, s, GM_FC, &a, 1, 0, H / 128, c.n_fused * H, tm_feats, R, p, true, 1, DFLASH_KID_FC);
    if (rc) return rc;
  }

  if (target) {  // pages for the block's positions (the context length moves with dflash_advance)
    h->launches++;
    rc = cuda_err(launch_page_alloc(slots, batch, DFL_BLOCK, nullptr, DFL_BLOCK, h->ctx_len, h->pos0, h->n_pages,
                                    h->page_table, c.max_pages_per_slot, h->free_stack, h->free_top, h->n_eff,
                                    h->slots_ok, c.max_slots, h->status, s));
    if (rc) return rc;
  }
  h->launches++;
  BlockCtx bcx;
  bcx.ctx_len = h->ctx_len;
  bcx.page_table = h->page_table;
  bcx.max_pages_per_slot = c.max_pages_per_slot;
  bcx.max_pages = c.max_pages;
  bcx.rope = h->rope;
  bcx.D = D;
  bcx.max_pos = h->max_pos;
  bcx.block = c.block;
  bcx.bctx = h->bctx;
  bcx.tokens = vf.tokens;
  bcx.n_valid = vf.n_valid;
  bcx.slots_ok = h->slots_ok;
  bcx.max_slots = c.max_slots;
  bcx.brope = h->brope;
  // with several requests, the attention grid takes them longest first: its
  // CTAs start in grid order, so the short requests fill the last wave
  bcx.order = batch > 1 ? h->attn_order : nullptr;
  rc = cuda_err(launch_embed(slots, batch, last_tok, c.mask_id, c.vocab, h->embed_pk, h->embed_sc, h->in_norm[0], H, h->h,
                             h->hg, h->ss_a, h->keys, bcx, h->status, s));
  if (rc) return rc;

  for (int l = 0; l < c.n_layers; ++l) {
    {  // QKV projection + q/k norm + RoPE; block K/V into the cache
      GemmParams p = {};
      p.ss_in = h->ss_a;
      p.ss_parts = H / 128;
      p.out = h->qbuf;
      p.qn_gain = h->q_norm[l];
      p.kn_gain[0] = h->k_norm[l];
      p.layer = l;
      p.kv = kv;
      p.slots = h->slots_ok;
      p.ctx_len = h->ctx_len;
      p.bctx = h->bctx;
      p.brope = h->brope;
      p.rows_per_req = DFL_BLOCK;
      p.N = (hq + 2 * hkv) * D;
      if (fold) {
        p.ss_ld = M;
        p.inj_m0 = M;
        p.ss_inj = h->ss_c;
        p.inj_ld = R;
        p.rows_per_req = rows_per_req;
        p.pos0 = h->pos0;
        p.n_eff = h->n_eff;
      }
      const void* a = h->wqkv_pk[l];
      fp8_weights(h, p, h->wqkv_sc[l]);
      rc = run_gemm(h, s, GM_QKV, &a, 1, 0, p.N / 128, H, fold ? h->tm_hgx : h->tm_hg_s, fold ? M + R : M, p, true, 0,
                    DFLASH_KID_QKV, fold ? DFL_BN_MAX : bn_small(M));
      if (rc) return rc;
    }
    {  // block attention
      AttnParams a = {};
      a.q = h->qbuf;
      a.out = h->obuf;
      a.kv = kv;
      a.layer = l;
      a.slots = h->slots_ok;
      a.ctx_len = h->ctx_len;
      a.hq = hq;
      a.hkv = hkv;
      a.D = D;
      a.n_splits = h->attn_splits;
      a.merge_global = h->attn_global ? 1 : 0;
      a.part = h->attn_part;
      a.block = c.block;
      a.causal = target ? 1 : 0;
      a.n_valid = vf.n_valid;
      a.order = batch > 1 ? h->attn_order : nullptr;
      a.early = fold ? 0 : 1;  // a folded QKV projection appends context rows itself
      a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D));
      a.status = h->status;
      if (unsigned long long* tb = h->trace.take(DFLASH_KID_ATTENTION, (long long)a.n_splits * hkv * batch))
        a.trace = tb;
      ProbeScope ps(h, DFLASH_KID_ATTENTION, s);
      h->launches++;
      rc = cuda_err(attn_launch(a, batch, s, h->pdl, h->attn_tc));
      if (rc) return rc;
    }
    {  // output projection + residual; post-attention norm inputs
      GemmParams p = {};
      p.h = h->h;
      p.out = h->hg;
      p.gain = h->post_norm[l];
      p.ss_out = h->ss_a;
      p.N = H;
      const void* a = h->wo_pk[l];
      fp8_weights(h, p, h->wo_sc[l]);
      rc = run_gemm(h, s, GM_RESID, &a, 1, 0, H / 128, hq * D, h->tm_o, M, p, true, 0, DFLASH_KID_WO);
      if (rc) return rc;
    }
    {  // gate/up projection + SiLU gating
      GemmParams p = {};
      p.ss_in = h->ss_a;
      p.ss_parts = H / 128;
      p.out = h->act;
      p.N = I;
      const void* a = h->gu_pk[l];
      fp8_weights(h, p, h->gu_sc[l]);
      rc = run_gemm(h, s, GM_SWIGLU, &a, 1, 0, I / 64, H, h->tm_hg, M, p, true, 0, DFLASH_KID_GATE_UP);
      if (rc) return rc;
    }
    {  // down projection + residual; next norm inputs
      GemmParams p = {};
      p.h = h->h;
      p.out = h->hg;
      p.gain = (l + 1 < c.n_layers) ? h->in_norm[l + 1] : h->final_norm;
      p.ss_out = h->ss_a;
      p.N = H;
      const void* a = h->down_pk[l];
      fp8_weights(h, p, h->down_sc[l]);
      rc = run_gemm(h, s, GM_RESID, &a, 1, 0, H / 128, I, h->tm_act, M, p, true, 0, DFLASH_KID_DOWN);
      if (rc) return rc;
    }
    if (vf.feats) {  // this layer's output is one of the drafter's fused features
      for (int k = 0; k < c.n_fused; ++k)
        if (tap_layer(k, c.n_layers, c.n_fused) == l) {
          h->launches++;
          rc = cuda_err(launch_tap(h->h, M, H, vf.feats, k, c.n_fused, s));
          if (rc) return rc;
        }
    }
  }
  if (hidden) {
    rc = cuda_err(cudaMemcpyAsync(hidden, h->h, (size_t)M * H * sizeof(float), cudaMemcpyDeviceToDevice, s));
    if (rc) return rc;
  }
  {  // final norm + tied lm_head + argmax
    GemmParams p = {};
    p.ss_in = h->ss_a;
    p.ss_parts = H / 128;
    p.N = c.vocab;
    p.keys = h->keys;
    p.logits = logits;
    p.draft = draft;
    p.block = c.block;
    p.row0 = target ? 0 : 1;
    p.temp_inv = smp.temp_inv;
    p.seed = smp.seed;
    p.round = smp.round;
    p.slots = h->slots_ok;  // a target's draws are keyed by slot and position
    p.bctx = h->bctx;
    p.done_ctr = h->done_ctr;
    const void* a = h->embed_pk;
    fp8_weights(h, p, h->embed_sc);
    rc = run_gemm(h, s, GM_ARGMAX, &a, 1, 0, ceil_div(c.vocab, 128), H, h->tm_hg, M, p, true, 0,
                  DFLASH_KID_LM_HEAD);
    if (rc) return rc;
  }
  return DFLASH_OK;
}

}  // namespace

extern "C" {

const char* dflash_status_string(int st) {
  switch (st) {
    case DFLASH_OK: return "ok";
    case DFLASH_ERR_INVALID_ARG: return "invalid argument";
    case DFLASH_ERR_SHAPE: return "unsupported shape";
    case DFLASH_ERR_CAPACITY: return "capacity exceeded";
    case DFLASH_ERR_CUDA: return "CUDA error";
    case DFLASH_ERR_DEVICE: return "device-side check failed";
    case DFLASH_ERR_WORKSPACE: return "workspace too small or misaligned";
    case DFLASH_ERR_RANGE: return "a weight exceeds the f16 range";
  }
  return "unknown status";
}

size_t dflash_workspace_bytes(const dflash_config* cfg) {
  if (!cfg_valid(cfg)) return 0;
  int sms = device_sms(cfg->device);
  if (sms <= 0) sms = 160;  // no device visible: size for the largest part
  return carve(nullptr, *cfg, nullptr, sms);
}

int dflash_create(const dflash_config* cfg, const dflash_weights* w, void* workspace, size_t bytes,
                  dflash_handle** out) {
  if (!out) return DFLASH_ERR_INVALID_ARG;
  *out = nullptr;
  if (!cfg_valid(cfg)) return DFLASH_ERR_SHAPE;
  const bool drafter = cfg->role == 0;  // a target has no fusion weights
  if (!w || !w->embed || (drafter && (!w->fc || !w->fc_norm)) || !w->final_norm || !w->in_norm || !w->wqkv ||
      !w->q_norm || !w->k_norm || !w->wo || !w->post_norm || !w->w_gate_up || !w->w_down)
    return DFLASH_ERR_INVALID_ARG;
  for (int l = 0; l < cfg->n_layers; ++l)
    if (!w->in_norm[l] || !w->wqkv[l] || !w->q_norm[l] || !w->k_norm[l] || !w->wo[l] || !w->post_norm[l] ||
        !w->w_gate_up[l] || !w->w_down[l])
      return DFLASH_ERR_INVALID_ARG;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255)) return DFLASH_ERR_WORKSPACE;
  if (cudaSetDevice(cfg->device) != cudaSuccess) return DFLASH_ERR_CUDA;
  const int sms = device_sms(cfg->device);
  if (sms <= 0) return DFLASH_ERR_CUDA;
  if (bytes < carve(nullptr, *cfg, nullptr, sms)) return DFLASH_ERR_WORKSPACE;
  if (!load_encode()) return DFLASH_ERR_CUDA;

  dflash_handle* h = new (std::nothrow) dflash_handle();
  if (!h) return DFLASH_ERR_CAPACITY;
  h->cfg = *cfg;
  h->num_sms = sms;
  h->fp8 = cfg->weight_fp8 != 0;
  const size_t need = carve(h, *cfg, static_cast<char*>(workspace), sms);
  if (cuda_err(cudaMemset(workspace, 0, need))) {
    delete h;
    return DFLASH_ERR_CUDA;
  }
  const dflash_config& c = *cfg;
  const int H = c.hidden, D = c.head_dim, hq = c.n_q_heads, hkv = c.n_kv_heads, I = c.intermediate;
  auto B16 = [](const void* p) { return static_cast<const bf16*>(p); };
  // f16 packing, or FP8 E4M3 packing with per-row scales
  auto pack = [&](const void* src, f16* dst, float* sc, int N, int K, int n_tiles, int swiglu_I) {
    return h->fp8 ? launch_pack_weight_fp8(B16(src), reinterpret_cast<uint8_t*>(dst), sc, N, K, n_tiles, swiglu_I, 0)
                  : launch_pack_weight(B16(src), dst, N, K, n_tiles, swiglu_I, true, h->status, 0);
  };
  cudaError_t e = pack(w->embed, h->embed_pk, h->embed_sc, c.vocab, H, ceil_div(c.vocab, 128), 0);
  if (!e && drafter) e = launch_pack_weight(B16(w->fc), h->fc_pk, H, c.n_fused * H, H / 128, 0, false, h->status, 0);
  if (!e && drafter) e = launch_gain_f32(B16(w->fc_norm), h->fc_norm, H, 0);
  if (!e) e = launch_gain_f32(B16(w->final_norm), h->final_norm, H, 0);
  for (int l = 0; l < c.n_layers && !e; ++l) {
    e = pack(w->wqkv[l], h->wqkv_pk[l], h->wqkv_sc[l], (hq + 2 * hkv) * D, H, (hq + 2 * hkv) * D / 128, 0);
    if (!e) e = pack(w->wo[l], h->wo_pk[l], h->wo_sc[l], H, hq * D, H / 128, 0);
    if (!e) e = pack(w->w_gate_up[l], h->gu_pk[l], h->gu_sc[l], 2 * I, H, I / 64, I);
    if (!e) e = pack(w->w_down[l], h->down_pk[l], h->down_sc[l], H, I, H / 128, 0);
    if (!e) e = launch_gain_f32(B16(w->in_norm[l]), h->in_norm[l], H, 0);
    if (!e) e = launch_gain_f32(B16(w->post_norm[l]), h->post_norm[l], H, 0);
    if (!e) e = launch_gain_f32(B16(w->q_norm[l]), h->q_norm[l], D, 0);
    if (!e) e = launch_gain_f32(B16(w->k_norm[l]), h->k_norm[l], D, 0);
  }
  bool ok = e == cudaSuccess;
  int rc = ok ? DFLASH_OK : DFLASH_ERR_CUDA;
  if (!rc) rc = cuda_err(gemm_init_attributes());
  if (!rc) rc = cuda_err(attn_init_attributes());
  // token tiles of 128+ tokens: clusters of 4 CTAs share each tile unless
  // pairs keep clearly more SMs busy (clusters are placed within one GPC)
  if (!rc && DFL_GEMM_MAX_CL > 1) {
    const int st = gemm_pick_stages(DFL_BN_MAX, GM_QKV, 0);
    const int n2 = 2 * gemm_max_clusters(DFL_BN_MAX, st, 2);
    const int n4 = DFL_GEMM_MAX_CL >= 4 ? 4 * gemm_max_clusters(DFL_BN_MAX, st, 4) : 0;
    if (n4 > 0 && 10 * n4 >= 9 * n2) {
      h->gemm_cl = 4;
      h->gemm_cl_ctas = std::min(n4, sms);
    } else if (n2 > 0) {
      h->gemm_cl = 2;
      h->gemm_cl_ctas = std::min(n2, sms);
    }
  }
  // page loop: the tcgen05 one has the higher fixed cost per CTA and the
  // higher rate per page, so it is chosen when a split holds 8 pages or more
  // at full slot capacity (measured on GB300: slower at 4-5 pages per split,
  // faster at 11 -- 769.6 vs 775.2 us per Llama-3.1-8B-shaped round -- and at
  // 57-86)
  h->attn_tc = c.attn_impl == 2 || (c.attn_impl == 0 && ceil_div(c.max_pages_per_slot, h->attn_splits) >= 8);
  // every (request, KV head) cluster in one wave: a second wave would double
  // the attention time, so take the most splits whose clusters all fit
  while (!rc && h->attn_splits > 1 &&
         attn_max_active_clusters(c.head_dim, c.n_q_heads, c.n_kv_heads, h->attn_splits, h->attn_tc) <
             c.max_batch * c.n_kv_heads)
    --h->attn_splits;
  // more splits than clusters allow, each still holding 32+ pages at full
  // slot capacity: merge them through global memory instead (measured on
  // GB300: 9 splits of ~57 pages beat 6 clusters of ~86 by 83 us per
  // long-context round; 19 splits of ~8 pages lost 45 us to 12 clusters of
  // ~12 on the Llama-3.1-8B shape -- the second kernel and the per-CTA set-up
  // outweigh the shorter page loops)
  if (!rc && h->attn_part) {
    const int gs = global_attn_splits(c, sms);
    if (gs > h->attn_splits && ceil_div(c.max_pages_per_slot, gs) >= DFL_ATTN_GLOBAL_MIN_PAGES) {
      h->attn_global = true;
      h->attn_splits = gs;
      h->attn_tc = c.attn_impl == 2 || (c.attn_impl == 0 && ceil_div(c.max_pages_per_slot, gs) >= 8);
    }
  }
  if (!rc)
    rc = cuda_err(cudaMemset(h->page_table, 0xFF, (size_t)c.max_slots * c.max_pages_per_slot * sizeof(int)));
  if (!rc) rc = cuda_err(launch_pool_init(h->free_stack, h->free_top, c.max_pages, 0));
  if (!rc) rc = cuda_err(launch_rope_table(h->rope, h->max_pos, D, c.rope_theta, 0));
  if (!rc) rc = cuda_err(cudaDeviceSynchronize());
  if (!rc) {  // a weight the f16 copies cannot hold (the packing saturated it): refuse the handle
    uint32_t st = 0;
    rc = cuda_err(cudaMemcpy(&st, h->status, sizeof(st), cudaMemcpyDeviceToHost));
    if (!rc && (st & DFLASH_DEV_RANGE)) {
      fprintf(stderr, "[dflash] dflash_create: a weight exceeds the f16 range (|w| > 65504); "
                      "create the handle with weight_fp8 = 1 (per-row scales) instead\n");
      rc = DFLASH_ERR_RANGE;
    }
  }
  if (rc) {
    delete h;
    return rc;
  }
  *out = h;
  return DFLASH_OK;
}

int dflash_destroy(dflash_handle* h) {
  if (!h) return DFLASH_ERR_INVALID_ARG;
  if (h->exec) cudaGraphExecDestroy(h->exec);
  if (h->graph) cudaGraphDestroy(h->graph);
  for (cudaEvent_t e : h->probe.ev) cudaEventDestroy(e);
  for (cudaEvent_t e : h->marks.ev) cudaEventDestroy(e);
  delete h;
  return DFLASH_OK;
}

int dflash_fuse_inject(dflash_handle* h, const int32_t* slots, int32_t batch, const void* feats,
                       int32_t rows_per_req, const int32_t* n_new, void* stream) {
  if (!h || h->cfg.role != 0 || batch < 0 || batch > h->cfg.max_batch || rows_per_req < 0)
    return DFLASH_ERR_INVALID_ARG;
  if ((long long)batch * rows_per_req > h->cfg.max_rows) return DFLASH_ERR_CAPACITY;
  if (batch == 0) return DFLASH_OK;
  if (!slots || !n_new) return DFLASH_ERR_INVALID_ARG;
  if (rows_per_req > 0 && !feats) return DFLASH_ERR_INVALID_ARG;
  if (cudaSetDevice(h->cfg.device) != cudaSuccess) return DFLASH_ERR_CUDA;
  cudaStream_t s = (cudaStream_t)stream;
  const dflash_config& c = h->cfg;
  const int H = c.hidden, D = c.head_dim, hkv = c.n_kv_heads;
  const int R = batch * rows_per_req;
  // A round's injection over more rows than one token tile holds computes
  // only the appended rows: they are gathered densely first, and the GEMMs
  // read their count on the device.
  const bool compact = R > DFL_BN_MAX && rows_per_req <= DFL_BLOCK && h->cstage;
  // every descriptor is encoded (and the caller's feature rows checked:
  // 16-byte aligned) before anything is queued, so a refused call leaves the
  // slots' lengths and pages untouched
  CUtensorMap tm_feats;
  if (R > 0) {
    const uint32_t BN = gemm_shape(h, R, bn_small(R)).box();
    if (!make_tmap(&tm_feats, feats, R, (uint64_t)c.n_fused * H, BN, true)) return DFLASH_ERR_INVALID_ARG;
    if (h->bm_rows != R) {
      if (!make_tmap(&h->tm_cg, h->cg, R, H, BN)) return DFLASH_ERR_CUDA;
      h->bm_rows = R;
    }
    if (compact && h->bm_cstage != R) {
      if (!make_tmap(&h->tm_cstage, h->cstage, R, (uint64_t)c.n_fused * H, BN, true)) return DFLASH_ERR_CUDA;
      h->bm_cstage = R;
    }
  }
  h->launches++;
  int rc = cuda_err(launch_page_alloc(slots, batch, h->cfg.block, n_new, rows_per_req, h->ctx_len, h->pos0, h->n_pages,
                                      h->page_table, c.max_pages_per_slot, h->free_stack, h->free_top, h->n_eff, h->slots_ok,
                                      c.max_slots, h->status, s, compact ? h->row_off : nullptr,
                                      compact ? h->n_live : nullptr));
  if (rc || R == 0) return rc;
  if (compact) {
    h->launches++;
    rc = cuda_err(launch_compact_rows(static_cast<const bf16*>(feats), batch, rows_per_req, c.n_fused * H, h->n_eff,
                                      h->row_off, h->cstage, h->row_map, s));
    if (rc) return rc;
  }
  {  // fusion projection; RMSNorm gain folded in, its scale deferred to the consumer
    GemmParams p = {};
    p.out = h->cg;
    p.gain = h->fc_norm;
    p.ss_out = h->ss_c;
    p.N = H;
    if (compact) p.m_dyn = h->n_live;
    const void* a = h->fc_pk;
    rc = run_gemm(h, s, GM_FC, &a, 1, 0, H / 128, c.n_fused * H, compact ? h->tm_cstage : tm_feats, R, p, true, 1,
                  DFLASH_KID_FC, bn_small(R));
    if (rc) return rc;
  }
  {  // every layer's K/V projection of the fused feature, k-norm, RoPE, paged append
    GemmParams p = {};
    p.ss_in = h->ss_c;
    p.ss_parts = H / 128;
    p.N = 2 * hkv * D;
    for (int l = 0; l < c.n_layers; ++l) p.kn_gain[l] = h->k_norm[l];
    p.kv = kv_geom(h);
    p.slots = h->slots_ok;
    p.pos0 = h->pos0;
    p.n_eff = h->n_eff;
    p.rows_per_req = rows_per_req;
    if (compact) {
      p.m_dyn = h->n_live;
      p.row_map = h->row_map;
    }
    const void* a[DFL_MAX_LAYERS];
    for (int l = 0; l < c.n_layers; ++l) {
      a[l] = h->wqkv_pk[l];
      fp8_weights(h, p, h->wqkv_sc[l], l);
    }
    rc = run_gemm(h, s, GM_INJECT, a, c.n_layers, c.n_q_heads * D / 128, p.N / 128, H, h->tm_cg, R, p, true, 0,
                  DFLASH_KID_INJECT, bn_small(R));
    if (rc) return rc;
  }
  return DFLASH_OK;
}

int dflash_draft_block(dflash_handle* h, const int32_t* slots, int32_t batch, const int32_t* last_tok,
                       int32_t* draft, void* stream) {
  return draft_impl(h, slots, batch, last_tok, draft, nullptr, nullptr, stream);
}

int dflash_draft_round(dflash_handle* h, const int32_t* slots, int32_t batch, const void* feats,
                       int32_t rows_per_req, const int32_t* n_new, const int32_t* last_tok, int32_t* draft,
                       void* stream) {
  if (!h || h->cfg.role != 0 || batch < 0 || batch > h->cfg.max_batch || rows_per_req < 0)
    return DFLASH_ERR_INVALID_ARG;
  if (batch == 0) return DFLASH_OK;
  // folding needs the feature rows to fit below the block rows in one token tile
  const long long R = (long long)batch * rows_per_req;
  if (rows_per_req == 0 || rows_per_req > DFL_BLOCK || batch * DFL_BLOCK + R > DFL_BN_MAX || R > h->cfg.max_rows) {
    int rc = dflash_fuse_inject(h, slots, batch, feats, rows_per_req, n_new, stream);
    if (rc) return rc;
    return draft_impl(h, slots, batch, last_tok, draft, nullptr, nullptr, stream);
  }
  if (!slots || !n_new || !feats) return DFLASH_ERR_INVALID_ARG;
  return draft_impl(h, slots, batch, last_tok, draft, nullptr, nullptr, stream, feats, rows_per_req, n_new);
}

int dflash_draft_block_debug(dflash_handle* h, const int32_t* slots, int32_t batch, const int32_t* last_tok,
                             int32_t* draft, float* hidden, float* logits, void* stream) {
  return draft_impl(h, slots, batch, last_tok, draft, hidden, logits, stream);
}

int dflash_verify_block(dflash_handle* h, const int32_t* slots, int32_t batch, const int32_t* tokens,
                        const int32_t* n_valid, int32_t* out_tok, void* feats, void* stream) {
  if (!h || h->cfg.role != 1 || !tokens || !out_tok) return DFLASH_ERR_INVALID_ARG;
  Verify vf;
  vf.tokens = tokens;
  vf.n_valid = n_valid;
  vf.feats = static_cast<bf16*>(feats);
  return draft_impl(h, slots, batch, nullptr, out_tok, nullptr, nullptr, stream, nullptr, 0, nullptr, Sampling(), vf);
}

int dflash_verify_block_sample(dflash_handle* h, const int32_t* slots, int32_t batch, const int32_t* tokens,
                               const int32_t* n_valid, float temperature, uint64_t seed, int32_t* out_tok, void* feats,
                               void* stream) {
  if (!h || h->cfg.role != 1 || !tokens || !out_tok) return DFLASH_ERR_INVALID_ARG;
  if (!(temperature == temperature) || temperature < 0.f) return DFLASH_ERR_INVALID_ARG;
  Verify vf;
  vf.tokens = tokens;
  vf.n_valid = n_valid;
  vf.feats = static_cast<bf16*>(feats);
  Sampling smp;
  smp.temp_inv = temperature >= 1e-6f ? 1.f / temperature : 0.f;  // below: the draw is the argmax
  smp.seed = seed;
  return draft_impl(h, slots, batch, nullptr, out_tok, nullptr, nullptr, stream, nullptr, 0, nullptr, smp, vf);
}

int dflash_advance(dflash_handle* h, const int32_t* slots, int32_t batch, const int32_t* n, void* stream) {
  if (!h || batch < 0 || batch > h->cfg.max_batch) return DFLASH_ERR_INVALID_ARG;
  if (batch == 0) return DFLASH_OK;
  if (!slots || !n) return DFLASH_ERR_INVALID_ARG;
  if (cudaSetDevice(h->cfg.device) != cudaSuccess) return DFLASH_ERR_CUDA;
  const dflash_config& c = h->cfg;
  h->launches++;
  return cuda_err(launch_page_alloc(slots, batch, DFL_BLOCK, n, DFL_BLOCK, h->ctx_len, h->pos0, h->n_pages,
                                    h->page_table, c.max_pages_per_slot, h->free_stack, h->free_top, h->n_eff,
                                    h->slots_ok, c.max_slots, h->status, (cudaStream_t)stream));
}

int dflash_draft_block_sample(dflash_handle* h, const int32_t* slots, int32_t batch, const int32_t* last_tok,
                              float temperature, uint64_t seed, const int32_t* round, int32_t* draft, float* logits,
                              void* stream) {
  if (!(temperature == temperature) || temperature < 0.f) return DFLASH_ERR_INVALID_ARG;
  Sampling smp;
  smp.temp_inv = temperature >= 1e-6f ? 1.f / temperature : 0.f;  // below: the draw is the argmax
  smp.seed = seed;
  smp.round = round;
  return draft_impl(h, slots, batch, last_tok, draft, nullptr, logits, stream, nullptr, 0, nullptr, smp);
}

int dflash_accept_trim(dflash_handle* h, const int32_t* slots, int32_t batch, const int32_t* draft,
                       const int32_t* target, int32_t* accept_len, int32_t* bonus, int32_t* ctx_len,
                       void* stream) {
  if (!h || batch < 0 || batch > h->cfg.max_batch) return DFLASH_ERR_INVALID_ARG;
  if (batch == 0) return DFLASH_OK;
  if (!slots || !draft || !target || !accept_len || !bonus || !ctx_len) return DFLASH_ERR_INVALID_ARG;
  if (cudaSetDevice(h->cfg.device) != cudaSuccess) return DFLASH_ERR_CUDA;
  h->launches++;
  return cuda_err(launch_accept(slots, batch, h->cfg.block, draft, target, accept_len, bonus, ctx_len, h->ctx_len,
                                h->cfg.max_slots, h->status, (cudaStream_t)stream));
}

int dflash_check_wait_timeout(dflash_handle* h, uint32_t limit_us, void* stream) {
  if (!h || limit_us < 1 || limit_us > 100000) return DFLASH_ERR_INVALID_ARG;
  if (cudaSetDevice(h->cfg.device) != cudaSuccess) return DFLASH_ERR_CUDA;
  h->launches++;
  return cuda_err(launch_wait_check(h->status, (unsigned long long)limit_us * 1000ull, (cudaStream_t)stream));
}

int dflash_reset_slot(dflash_handle* h, int32_t slot, void* stream) {
  if (!h || slot < 0 || slot >= h->cfg.max_slots) return DFLASH_ERR_INVALID_ARG;
  if (cudaSetDevice(h->cfg.device) != cudaSuccess) return DFLASH_ERR_CUDA;
  h->launches++;
  return cuda_err(launch_reset_slot(slot, h->ctx_len, h->n_pages, h->page_table, h->cfg.max_pages_per_slot,
                                    h->free_stack, h->free_top, (cudaStream_t)stream));
}

int dflash_read_status(dflash_handle* h, uint32_t* out) {
  if (!h || !out) return DFLASH_ERR_INVALID_ARG;
  if (cudaSetDevice(h->cfg.device) != cudaSuccess) return DFLASH_ERR_CUDA;
  int rc = cuda_err(cudaDeviceSynchronize());
  if (rc) return rc;
  rc = cuda_err(cudaMemcpy(out, h->status, sizeof(uint32_t), cudaMemcpyDeviceToHost));
  if (rc) return rc;
  return cuda_err(cudaMemset(h->status, 0, sizeof(uint32_t)));
}

int dflash_graph_begin(dflash_handle* h, void* stream) {
  if (!h) return DFLASH_ERR_INVALID_ARG;
  if (cudaSetDevice(h->cfg.device) != cudaSuccess) return DFLASH_ERR_CUDA;
  return cuda_err(cudaStreamBeginCapture((cudaStream_t)stream, cudaStreamCaptureModeThreadLocal));
}

int dflash_graph_end(dflash_handle* h, void* stream, int32_t* n_kernels) {
  if (!h) return DFLASH_ERR_INVALID_ARG;
  cudaGraph_t g = nullptr;
  int rc = cuda_err(cudaStreamEndCapture((cudaStream_t)stream, &g));
  if (rc) return rc;
  size_t n = 0;
  rc = cuda_err(cudaGraphGetNodes(g, nullptr, &n));
  std::vector<cudaGraphNode_t> nodes(n);
  if (!rc && n) rc = cuda_err(cudaGraphGetNodes(g, nodes.data(), &n));
  int kernels = 0;
  for (size_t i = 0; i < n && !rc; ++i) {
    cudaGraphNodeType t;
    if (cudaGraphNodeGetType(nodes[i], &t) == cudaSuccess && t == cudaGraphNodeTypeKernel) ++kernels;
  }
  cudaGraphExec_t e = nullptr;
  if (!rc) rc = cuda_err(cudaGraphInstantiate(&e, g, 0));
  if (!rc) rc = cuda_err(cudaGraphUpload(e, (cudaStream_t)stream));
  if (rc) {
    if (e) cudaGraphExecDestroy(e);
    if (g) cudaGraphDestroy(g);
    return rc;
  }
  if (h->exec) cudaGraphExecDestroy(h->exec);
  if (h->graph) cudaGraphDestroy(h->graph);
  h->graph = g;
  h->exec = e;
  if (n_kernels) *n_kernels = kernels;
  return DFLASH_OK;
}

int dflash_graph_launch(dflash_handle* h, void* stream) {
  if (!h || !h->exec) return DFLASH_ERR_INVALID_ARG;
  return cuda_err(cudaGraphLaunch(h->exec, (cudaStream_t)stream));
}

int dflash_read_kv(dflash_handle* h, int32_t layer, int32_t slot, int32_t pos0, int32_t n, void* k_out,
                   void* v_out, void* stream) {
  if (!h || !k_out || !v_out || layer < 0 || layer >= h->cfg.n_layers || slot < 0 || slot >= h->cfg.max_slots ||
      pos0 < 0 || n < 0 || pos0 + n > h->max_pos)
    return DFLASH_ERR_INVALID_ARG;
  if (cudaSetDevice(h->cfg.device) != cudaSuccess) return DFLASH_ERR_CUDA;
  return cuda_err(launch_read_kv(kv_geom(h), layer, slot, pos0, n, static_cast<float*>(k_out),
                                 static_cast<float*>(v_out), (cudaStream_t)stream));
}

int dflash_slot_lengths(dflash_handle* h, const int32_t* slots, int32_t batch, int32_t* out, void* stream) {
  if (!h || batch < 0) return DFLASH_ERR_INVALID_ARG;
  if (batch == 0) return DFLASH_OK;
  if (!slots || !out) return DFLASH_ERR_INVALID_ARG;
  if (cudaSetDevice(h->cfg.device) != cudaSuccess) return DFLASH_ERR_CUDA;
  return cuda_err(launch_slot_lengths(slots, batch, h->ctx_len, h->cfg.max_slots, out, (cudaStream_t)stream));
}

int dflash_probe_arm(dflash_handle* h, int32_t kernel_id, int32_t n) {
  if (!h || n < 0) return DFLASH_ERR_INVALID_ARG;
  if (cudaSetDevice(h->cfg.device) != cudaSuccess) return DFLASH_ERR_CUDA;
  while ((int)h->probe.ev.size() < 2 * n) {
    cudaEvent_t e;
    int rc = cuda_err(cudaEventCreate(&e));
    if (rc) return rc;
    h->probe.ev.push_back(e);
  }
  h->probe.kid = kernel_id;
  h->probe.n = n;
  h->probe.next = 0;
  return DFLASH_OK;
}

int dflash_probe_read(dflash_handle* h, float* ms_out, int32_t cap, int32_t* n_out) {
  if (!h || (!ms_out && cap > 0)) return DFLASH_ERR_INVALID_ARG;
  const int n = std::min(h->probe.next, (int)cap);
  for (int i = 0; i < n; ++i) {
    int rc = cuda_err(cudaEventSynchronize(h->probe.ev[2 * i + 1]));
    if (rc) return rc;
    rc = cuda_err(cudaEventElapsedTime(ms_out + i, h->probe.ev[2 * i], h->probe.ev[2 * i + 1]));
    if (rc) return rc;
  }
  if (n_out) *n_out = n;
  return DFLASH_OK;
}

int dflash_marks_arm(dflash_handle* h, int32_t n) {
  if (!h || n < 0) return DFLASH_ERR_INVALID_ARG;
  if (cudaSetDevice(h->cfg.device) != cudaSuccess) return DFLASH_ERR_CUDA;
  while ((int)h->marks.ev.size() < n) {
    cudaEvent_t e;
    int rc = cuda_err(cudaEventCreate(&e));
    if (rc) return rc;
    h->marks.ev.push_back(e);
  }
  h->marks.n = n;
  h->marks.next = 0;
  return DFLASH_OK;
}

int dflash_mark(dflash_handle* h, void* stream) {
  if (!h) return DFLASH_ERR_INVALID_ARG;
  if (h->marks.next >= h->marks.n) return DFLASH_OK;
  if (cudaSetDevice(h->cfg.device) != cudaSuccess) return DFLASH_ERR_CUDA;
  cudaStream_t s = (cudaStream_t)stream;
  cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
  const bool capturing = cudaStreamIsCapturing(s, &st) == cudaSuccess && st == cudaStreamCaptureStatusActive;
  cudaEvent_t e = h->marks.ev[h->marks.next++];
  return cuda_err(capturing ? cudaEventRecordWithFlags(e, s, cudaEventRecordExternal) : cudaEventRecord(e, s));
}

int dflash_marks_read(dflash_handle* h, float* ms_out, int32_t cap, int32_t* n_out) {
  if (!h || (!ms_out && cap > 0)) return DFLASH_ERR_INVALID_ARG;
  const int n = std::min(h->marks.next - 1, (int)cap);
  for (int i = 0; i < n; ++i) {
    int rc = cuda_err(cudaEventSynchronize(h->marks.ev[i + 1]));
    if (rc) return rc;
    rc = cuda_err(cudaEventElapsedTime(ms_out + i, h->marks.ev[i], h->marks.ev[i + 1]));
    if (rc) return rc;
  }
  if (n_out) *n_out = n < 0 ? 0 : n;
  return DFLASH_OK;
}

uint64_t dflash_launch_count(dflash_handle* h) { return h ? h->launches : 0; }

int dflash_plan(dflash_handle* h, int32_t* out5) {
  if (!h || !out5) return DFLASH_ERR_INVALID_ARG;
  out5[0] = h->num_sms;
  out5[1] = h->attn_splits;
  out5[2] = h->attn_tc ? 2 : 1;
  out5[3] = h->gemm_cl;
  out5[4] = h->attn_global ? 1 : 0;
  return DFLASH_OK;
}

int dflash_trace_arm(dflash_handle* h, int32_t kernel_id, unsigned long long* buf, int32_t cap_ctas) {
  if (!h || (kernel_id && (!buf || cap_ctas <= 0))) return DFLASH_ERR_INVALID_ARG;
  h->trace.kid = kernel_id;
  h->trace.buf = buf;
  h->trace.cap = cap_ctas;
  h->trace.used = 0;
  return DFLASH_OK;
}

int dflash_harness_verify(dflash_handle* h, const int32_t* slots, int32_t batch, const int32_t* draft,
                          const int32_t* match, const int32_t* offs, int32_t rounds_cap, int32_t* round_ctr,
                          int32_t* target, const void* feat_stream, int32_t stream_rows, void* feats_out,
                          void* stream) {
  if (!h || batch < 0 || batch > h->cfg.max_batch) return DFLASH_ERR_INVALID_ARG;
  if (batch == 0) return DFLASH_OK;
  if (!slots || !draft || !match || !offs || !round_ctr || !target || rounds_cap <= 0) {
    return DFLASH_ERR_INVALID_ARG;
  }
  if (feat_stream && (!feats_out || stream_rows <= 0)) return DFLASH_ERR_INVALID_ARG;
  if (cudaSetDevice(h->cfg.device) != cudaSuccess) return DFLASH_ERR_CUDA;
  h->launches++;
  unsigned long long* stamp = nullptr;
  if (h->stamps && h->stamp_next < h->stamp_cap) stamp = h->stamps + 2 * (size_t)h->stamp_next++;
  return cuda_err(launch_harness_verify(slots, batch, h->cfg.block, draft, match, offs, rounds_cap, round_ctr, target,
                                        h->cfg.vocab, static_cast<const bf16*>(feat_stream), stream_rows,
                                        static_cast<bf16*>(feats_out), h->cfg.n_fused * h->cfg.hidden,
                                        h->ctx_len, h->cfg.max_slots, stamp, h->done_ctr + 8, (cudaStream_t)stream));
}

int dflash_stamps_arm(dflash_handle* h, unsigned long long* buf, int32_t n) {
  if (!h || n < 0 || (n > 0 && !buf)) return DFLASH_ERR_INVALID_ARG;
  h->stamps = n > 0 ? buf : nullptr;
  h->stamp_cap = n;
  h->stamp_next = 0;
  return DFLASH_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// dflash_fuse_inject_noalloc: dflash_fuse_inject with its per-call scratch in
// a fixed array compiled into the library instead of the handle's workspace.
//
// The scratch is the fusion GEMM's output rows (f16) with their sums of
// squares, and the split-K partial sums and tile counters of the two GEMMs.
// Limits: batch * rows_per_req <= 64 rows; the GEMMs run on at most 16 CTAs.
// Size: 16*2*256*128*4 (partials) + 64*8192*2 (rows) + 64*64*4 (sums) +
// 2*4096*4 (counters) bytes, about 5.1 MB, held by every device that loads
// the library until the process exits.
namespace {
constexpr int NA_MAX_ROWS = 64;
constexpr int NA_MAX_CTAS = 16;
constexpr size_t NA_PART_BYTES = (size_t)NA_MAX_CTAS * 2 * DFL_BN_MAX * 128 * sizeof(float);
constexpr size_t NA_ROWS_BYTES = (size_t)NA_MAX_ROWS * 8192 * sizeof(f16);
constexpr size_t NA_SS_BYTES = (size_t)(8192 / 128) * NA_MAX_ROWS * sizeof(float);
constexpr int NA_MAX_TILES = 4096;
constexpr size_t NA_CTR_BYTES = 2 * (size_t)NA_MAX_TILES * sizeof(unsigned);  // arrivals, finalisers done
constexpr size_t NA_BYTES = NA_PART_BYTES + NA_ROWS_BYTES + NA_SS_BYTES + NA_CTR_BYTES;
}  // namespace

static __device__ __align__(256) unsigned char g_noalloc_scratch[NA_BYTES];

namespace {
std::mutex g_na_mutex;
void* g_na_addr[64] = {};  // device address of g_noalloc_scratch, per device ordinal

// Device address of the static scratch on `dev` (the current device); looked
// up once per device.
int noalloc_scratch(int dev, char** out) {
  if (dev < 0 || dev >= 64) return DFLASH_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_na_mutex);
  if (!g_na_addr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) return cuda_err(e == cudaSuccess ? cudaErrorInvalidSymbol : e);
    g_na_addr[dev] = p;
  }
  *out = static_cast<char*>(g_na_addr[dev]);
  return DFLASH_OK;
}

int noalloc_gemm(dflash_handle* h, cudaStream_t s, int mode, const void* const* a, int groups, int a_tile_off,
                 int n_tiles, int K, const CUtensorMap& B, int M, GemmParams p, uint32_t ab_type, float* part,
                 unsigned* ctr) {
  const int BN = ((M + 15) / 16) * 16;  // M <= 64: one token tile
  p.mode = mode;
  p.M = M;
  if (!p.ss_ld) p.ss_ld = M;
  p.kblocks = K / 64;
  p.n_tiles = n_tiles;
  p.t_tiles = 1;
  p.BN = BN;
  p.groups = groups;
  for (int g = 0; g < groups; ++g) p.a[g] = a[g];
  p.a_tile_off = a_tile_off;
  p.ab_type = ab_type;
  p.total_tiles = groups * n_tiles;
  p.cl = 1;
  p.n_tg = n_tiles;
  p.total_ctiles = p.total_tiles;
  p.allow_split = 1;
  p.stages = gemm_pick_stages(BN, mode, p.a_fp8);
  p.red_items = gemm_red_items(BN, p.stages, p.a_fp8);
  int cols = 32;
  while (cols < 2 * BN) cols *= 2;
  p.tmem_cols = cols;
  p.status = h->status;
  p.ws = part;
  p.tile_ctr = ctr;
  p.tile_fin = ctr + NA_MAX_TILES;
  p.eps = h->cfg.rms_eps;
  p.H = h->cfg.hidden;
  p.hq = h->cfg.n_q_heads;
  p.hkv = h->cfg.n_kv_heads;
  p.D = h->cfg.head_dim;
  p.rope = h->rope;
  p.max_pos = h->max_pos;
  if (p.total_tiles > NA_MAX_TILES) return DFLASH_ERR_CAPACITY;
  const long long units = (long long)p.total_tiles * p.kblocks;
  const int grid = (int)std::min<long long>(units, NA_MAX_CTAS);
  if (units * (grid + 1) >= (1LL << 31)) return DFLASH_ERR_SHAPE;
  h->launches++;
  return cuda_err(gemm_launch(B, p, grid, s, h->pdl));
}
}  // namespace

extern "C" int dflash_fuse_inject_noalloc(dflash_handle* h, const int32_t* slots, int32_t batch, const void* feats,
                                          int32_t rows_per_req, const int32_t* n_new, void* stream) {
  if (!h || h->cfg.role != 0 || batch < 0 || batch > h->cfg.max_batch || rows_per_req < 0)
    return DFLASH_ERR_INVALID_ARG;
  if ((long long)batch * rows_per_req > NA_MAX_ROWS) {
    fprintf(stderr, "[dflash] dflash_fuse_inject_noalloc: %lld rows exceed its static scratch limit of %d\n",
            (long long)batch * rows_per_req, NA_MAX_ROWS);
    return DFLASH_ERR_CAPACITY;
  }
  if (batch == 0) return DFLASH_OK;
  if (!slots || !n_new) return DFLASH_ERR_INVALID_ARG;
  if (rows_per_req > 0 && !feats) return DFLASH_ERR_INVALID_ARG;
  if (cudaSetDevice(h->cfg.device) != cudaSuccess) return DFLASH_ERR_CUDA;
  char* base = nullptr;
  int rc = noalloc_scratch(h->cfg.device, &base);
  if (rc) return rc;
  float* part = reinterpret_cast<float*>(base);
  f16* rows = reinterpret_cast<f16*>(base + NA_PART_BYTES);
  float* ss = reinterpret_cast<float*>(base + NA_PART_BYTES + NA_ROWS_BYTES);
  unsigned* ctr = reinterpret_cast<unsigned*>(base + NA_PART_BYTES + NA_ROWS_BYTES + NA_SS_BYTES);

  cudaStream_t s = (cudaStream_t)stream;
  const dflash_config& c = h->cfg;
  const int H = c.hidden, D = c.head_dim, hkv = c.n_kv_heads;
  const int R = batch * rows_per_req;
  // descriptors first (and the caller's feature rows checked), so a refused
  // call queues nothing
  const uint32_t BN = (uint32_t)(((R + 15) / 16) * 16);
  CUtensorMap tm_feats, tm_rows;
  if (R > 0) {
    if (!make_tmap(&tm_feats, feats, R, (uint64_t)c.n_fused * H, BN, true)) return DFLASH_ERR_INVALID_ARG;
    if (!make_tmap(&tm_rows, rows, R, H, BN)) return DFLASH_ERR_CUDA;
  }
  // tile counters must start at zero (the kernels also leave them at zero)
  rc = cuda_err(cudaMemsetAsync(ctr, 0, NA_CTR_BYTES, s));
  if (rc) return rc;
  h->launches++;
  rc = cuda_err(launch_page_alloc(slots, batch, h->cfg.block, n_new, rows_per_req, h->ctx_len, h->pos0, h->n_pages,
                                  h->page_table, c.max_pages_per_slot, h->free_stack, h->free_top, h->n_eff, h->slots_ok,
                                  c.max_slots, h->status, s));
  if (rc || R == 0) return rc;
  {
    GemmParams p = {};
    p.out = rows;
    p.gain = h->fc_norm;
    p.ss_out = ss;
    p.N = H;
    const void* a = h->fc_pk;
    rc = noalloc_gemm(h, s, GM_FC, &a, 1, 0, H / 128, c.n_fused * H, tm_feats, R, p, 1, part, ctr);
    if (rc) return rc;
  }
  {
    GemmParams p = {};
    p.ss_in = ss;
    p.ss_parts = H / 128;
    p.N = 2 * hkv * D;
    for (int l = 0; l < c.n_layers; ++l) p.kn_gain[l] = h->k_norm[l];
    p.kv = kv_geom(h);
    p.slots = h->slots_ok;
    p.pos0 = h->pos0;
    p.n_eff = h->n_eff;
    p.rows_per_req = rows_per_req;
    const void* a[DFL_MAX_LAYERS];
    for (int l = 0; l < c.n_layers; ++l) {
      a[l] = h->wqkv_pk[l];
      fp8_weights(h, p, h->wqkv_sc[l], l);
    }
    rc = noalloc_gemm(h, s, GM_INJECT, a, c.n_layers, c.n_q_heads * D / 128, p.N / 128, H, tm_rows, R, p, 0, part,
                      ctr);
  }
  return rc;
}
