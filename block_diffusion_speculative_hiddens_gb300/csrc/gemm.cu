// Weight-streaming GEMM on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// out[t][n] = sum_k X[t][k] * W[n][k] for the drafter's projections.  The
// weight matrix is the 128-row A operand ("swap-AB"): at batch 1 the block has
// only 16 token rows, which become the MMA's N dimension (16..256), so one
// tcgen05.mma.cta_group::1 M=128 instruction covers 128 output features x all
// tokens, and the weights stream through shared memory exactly once.
//
// Weights are packed once at handle creation into 16 KB blocks of 128 rows x
// 64 columns, each already laid out as the 128-byte-swizzle image tcgen05
// reads (tiles of a matrix stored tile-major, k-blocks contiguous), so a
// stage's weight tile is one contiguous untiled bulk copy from HBM.
//
// Pipeline per CTA (persistent, one per SM, 192 threads):
//   warp 0  producer: one 16 KB bulk copy for the weight block and one TMA
//           tiled load (128-byte swizzle) for the BNx64 token tile per stage,
//           completion on an mbarrier;
//   warp 1  TMEM allocator and single-thread MMA issuer (4 x K=16 per stage),
//           double-buffered fp32 accumulators in TMEM;
//   warps 2-5 epilogue: tcgen05.ld -> registers -> fused epilogue.
//
// Work split: the (tile, 64-wide k-block) units are divided evenly over the
// grid (stream-K style), so every SM streams the same number of weight bytes.
// A tile cut between CTAs writes fp32 partials; the last CTA to arrive (device
// counter, no waiting) sums them in k order -- deterministic -- and runs the
// epilogue.  All waits are bounded (%globaltimer) and report through the
// status word instead of hanging.
#include "common.cuh"
#include "internal.h"

// Build-time tuning knobs (the defaults are the shipped configuration).
#ifndef DFL_GEMM_MAX_STAGES
#define DFL_GEMM_MAX_STAGES 12
#endif
#ifndef DFL_GEMM_L2_HINT
#define DFL_GEMM_L2_HINT 1
#endif
#ifndef DFL_GEMM_SAMPLING  // 0 compiles the lm_head's temperature > 0 draw out
#define DFL_GEMM_SAMPLING 1
#endif
#ifndef DFL_GEMM_RED_MAX  // most split-K part chunks (8 KB) landed at once outside the last segment
#define DFL_GEMM_RED_MAX 16
#endif
#ifndef DFL_GEMM_A_CHUNKS  // bulk copies per 16 KB weight block
#define DFL_GEMM_A_CHUNKS 1
#endif
#ifndef DFL_GEMM_PRODUCERS  // weight-streaming threads of tiles up to 64 tokens (1 or 2)
#define DFL_GEMM_PRODUCERS 2
#endif


namespace {

constexpr int A_STAGE_BYTES = 128 * 128;  // 128 rows x 64 16-bit values
constexpr int STG_BYTES = 32 * 128 * 4;   // epilogue staging: 32 tokens x 128 rows fp32
constexpr int RED_PARTS = 4;               // fewest split-K part chunks the reduction buffer holds
constexpr int RED_CHUNK = 16 * 128;        // floats of one part's 16-column chunk (8 KB)
constexpr int RED_BYTES = RED_PARTS * RED_CHUNK * 4;
constexpr int EPI_THREADS = 128;
constexpr int GEMM_THREADS = 192;       // producer, MMA, 4 epilogue warps
constexpr int CONV_THREADS = 64;        // FP8 kernels: 2 more warps convert the weight blocks
constexpr int GEMM_THREADS_FP8 = GEMM_THREADS + CONV_THREADS;

// Unit arithmetic is 32-bit: the host guarantees units * grid < 2^31.
DFL_DEV int unit_start(int c, int U, int G) { return c * U / G; }
// CTA whose unit range [unit_start(c), unit_start(c+1)) contains unit u.
DFL_DEV int cta_of_unit(int u, int U, int G) { return ((u + 1) * G + U - 1) / U - 1; }

// Work is scheduled in tiles of cl n-tiles sharing one token tile; rank cr
// of the cluster computes n-tile (tile group * cl + cr).  Scheduled tile ct
// -> the tile this CTA computes, or -1 for a rank past its group's last
// n-tile (it streams a copy of the last weight tile and finalises nothing).
// With cl = 1 the two numberings coincide.
// tl: token tiles scheduled (p.t_tiles, or fewer for a launch whose live
// token rows are counted on the device); tile ids keep the p.t_tiles layout.
//
// The token tile is the slowest index of the scheduled order: the clusters'
// contiguous unit ranges then put the token tiles of one n-tile group on
// clusters a quarter (for four token tiles) of the grid apart, which stream
// the same weight blocks at about the same time, so DRAM serves each once
// and L2 the rest (with the token tile fastest, one cluster ran the token
// tiles of a group back to back and re-read its weights from DRAM for each).
#ifndef DFL_GEMM_LAND_PIPE  // 1: a finaliser's next chunk of split-K parts lands during the current one
#define DFL_GEMM_LAND_PIPE 1
#endif
#ifndef DFL_GEMM_TT_SLOW
#define DFL_GEMM_TT_SLOW 1
#endif
DFL_DEV void sched_decode(const GemmParams& p, int ct, int tl, int& rest, int& tt) {
  if (DFL_GEMM_TT_SLOW) {
    const int ngr = p.groups * p.n_tg;
    rest = ct % ngr;
    tt = ct / ngr;
  } else {
    rest = ct / tl;
    tt = ct % tl;
  }
}
DFL_DEV int tile_of(const GemmParams& p, int ct, int cr, int tl) {
  int rest, tt;
  sched_decode(p, ct, tl, rest, tt);
  const int nt = (rest % p.n_tg) * p.cl + cr;
  return nt < p.n_tiles ? ((rest / p.n_tg) * p.n_tiles + nt) * p.t_tiles + tt : -1;
}

// Counter-based random numbers for drafting at temperature > 0: SplitMix64
// (Steele, Lea and Flood, OOPSLA 2014).  A stream key folds (seed, purpose 1
// = draft, request, round, block row); element v of the stream is
// mix(key + (v+1) * golden); its top 23 bits give u = (bits + 1/2) * 2^-23 in
// (0, 1), exact in float32, and the Gumbel variate -ln(-ln u).
constexpr unsigned long long SM64_GOLD = 0x9E3779B97F4A7C15ull;
DFL_DEV unsigned long long sm64_mix(unsigned long long z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}
DFL_DEV unsigned long long draft_stream_key(unsigned long long seed, int b, int rnd, int row) {
  unsigned long long k = sm64_mix(seed + SM64_GOLD);
  k = sm64_mix(k + SM64_GOLD * 2ull);  // purpose id 1: the drafter's draws
  k = sm64_mix(k + SM64_GOLD * (unsigned long long)(b + 1));
  k = sm64_mix(k + SM64_GOLD * (unsigned long long)(rnd + 1));
  return sm64_mix(k + SM64_GOLD * (unsigned long long)(row + 1));
}
// The target's draws at temperature > 0 (its verify step): the stream of
// (seed, purpose 2 = target, request slot, position of the block row), so a
// position's numbers do not depend on the block or round it falls in.
DFL_DEV unsigned long long target_stream_key(unsigned long long seed, int slot, int pos) {
  unsigned long long k = sm64_mix(seed + SM64_GOLD);
  k = sm64_mix(k + SM64_GOLD * 3ull);  // purpose id 2
  k = sm64_mix(k + SM64_GOLD * (unsigned long long)(slot + 1));
  return sm64_mix(k + SM64_GOLD * (unsigned long long)(pos + 1));
}
// Out of line: the greedy epilogue, run once per vocabulary tile, keeps its
// compact code (the instruction cache holds it across tiles).
__device__ __noinline__ float gumbel_at(unsigned long long key, int v) {
  const unsigned long long bits = sm64_mix(key + SM64_GOLD * (unsigned long long)(v + 1));
  const float u = ((float)(unsigned)(bits >> 41) + 0.5f) * 1.1920928955078125e-7f;  // 2^-23
  return -logf(-logf(u));
}

// Wait (bounded) until the tile counter at `addr` reaches `target`: the
// acquire load makes every arriver's part visible.  False after DFL_WAIT_NS
// (DFLASH_DEV_TIMEOUT set).
DFL_DEV bool wait_count(const unsigned* addr, unsigned target, uint32_t* status) {
  uint64_t t0 = 0;
  while (true) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(addr) : "memory");
    if (v >= target) return true;
    const uint64_t t = globaltimer();
    if (t0 == 0) {
      t0 = t;
    } else if (t - t0 > DFL_WAIT_NS) {
      dev_error(status, DFLASH_DEV_TIMEOUT);
      return false;
    }
  }
}

// Timeline stamps (p.trace non-null): 0 entry, 1 set-up done, 2 first weight
// stage landed, 3 last MMA issued, 4 epilogue done, 5 exit, 6 units (low 32
// bits) and the launch's CTA count (high 32 bits), 7 SM id.
DFL_DEV void trace_at(const GemmParams& p, int ev, unsigned long long v) {
  if (p.trace) p.trace[(size_t)blockIdx.x * 8 + ev] = v;
}

// A lane's head-norm gains: g[j] = gain[lane + 32 j] for the rows it holds
// (D = 64: g[0], g[1] only).
DFL_DEV void load_head_gain(const float* gain, int D, int lane, float* g) {
#pragma unroll
  for (int j = 0; j < 4; ++j) g[j] = lane + 32 * j < D ? gain[lane + 32 * j] : 0.f;
}

constexpr int EPI_TOK = 4;  // tokens per warp whose inputs are gathered together

// Head RMSNorm + RoPE on the values a warp holds for EPI_TOK tokens (lane
// holds rows lane, lane+32, lane+64, lane+96 of a 128-row tile); g from
// load_head_gain; c0/c1[q] are token q's (cos, sin) of RoPE frequencies lane
// and lane+32.  D = 128: one head, RoPE pairs (0,2), (1,3).  D = 64: two
// heads (rows 0-63, 64-127), pairs (0,1) and (2,3), frequency lane.  The
// norms' shuffle reductions of all tokens are interleaved, so the warp pays
// one reduction latency, not one per token.
DFL_DEV void head_norm_rope4(float (&x)[EPI_TOK][4], const float* g, const float2* c0, const float2* c1, int D,
                             float eps) {
  if (D == 128) {
    float ss[EPI_TOK];
#pragma unroll
    for (int q = 0; q < EPI_TOK; ++q) ss[q] = x[q][0] * x[q][0] + x[q][1] * x[q][1] + x[q][2] * x[q][2] + x[q][3] * x[q][3];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
      for (int q = 0; q < EPI_TOK; ++q) ss[q] += __shfl_xor_sync(0xffffffffu, ss[q], o);
#pragma unroll
    for (int q = 0; q < EPI_TOK; ++q) {
      const float inv = rsqrtf(ss[q] / 128.f + eps);
#pragma unroll
      for (int j = 0; j < 4; ++j) x[q][j] *= inv * g[j];
      const float a0 = x[q][0], b0 = x[q][2], a1 = x[q][1], b1 = x[q][3];
      x[q][0] = a0 * c0[q].x - b0 * c0[q].y;
      x[q][2] = b0 * c0[q].x + a0 * c0[q].y;
      x[q][1] = a1 * c1[q].x - b1 * c1[q].y;
      x[q][3] = b1 * c1[q].x + a1 * c1[q].y;
    }
  } else {  // D == 64
    float sa[EPI_TOK], sb[EPI_TOK];
#pragma unroll
    for (int q = 0; q < EPI_TOK; ++q) {
      sa[q] = x[q][0] * x[q][0] + x[q][1] * x[q][1];
      sb[q] = x[q][2] * x[q][2] + x[q][3] * x[q][3];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
      for (int q = 0; q < EPI_TOK; ++q) {
        sa[q] += __shfl_xor_sync(0xffffffffu, sa[q], o);
        sb[q] += __shfl_xor_sync(0xffffffffu, sb[q], o);
      }
#pragma unroll
    for (int q = 0; q < EPI_TOK; ++q) {
      const float ia = rsqrtf(sa[q] / 64.f + eps), ib = rsqrtf(sb[q] / 64.f + eps);
      x[q][0] *= ia * g[0];
      x[q][1] *= ia * g[1];
      x[q][2] *= ib * g[0];
      x[q][3] *= ib * g[1];
      const float a0 = x[q][0], b0 = x[q][1], a1 = x[q][2], b1 = x[q][3];
      x[q][0] = a0 * c0[q].x - b0 * c0[q].y;
      x[q][1] = b0 * c0[q].x + a0 * c0[q].y;
      x[q][2] = a1 * c0[q].x - b1 * c0[q].y;
      x[q][3] = b1 * c0[q].x + a1 * c0[q].y;
    }
  }
}

// Page of position `pos` of `slot`, or -1 when it has none.
DFL_DEV int page_of(const GemmParams& p, int slot, int pos) {
  const int pi = pos >> 6;
  if (pi >= p.kv.max_pages_per_slot) return -1;
  const int pg = p.kv.page_table[(size_t)slot * p.kv.max_pages_per_slot + pi];
  return (pg < 0 || pg >= p.kv.max_pages) ? -1 : pg;
}


// Per-token inputs of a token tile, built once per token tile in shared
// memory by the epilogue warps while the main loop streams (so the tile's
// finalisation finds them there instead of waiting on dependent global
// loads): the RMSNorm scale of the GEMM's input and, for QKV/INJECT, the
// row's position, the page holding it (-1: none, -2: a padding row of a
// smaller block) and flags (bit 0: the row is written, bit 1: a fused-feature
// row -- QKV's folded injection rows, every INJECT row).
struct TokTab {
  float* s;
  int* pos;
  int* pg;
  int* flag;
};
constexpr int TOKTAB_BYTES = DFL_BN_MAX * 16;

template <int MODE>
DFL_DEV void build_toktab(const GemmParams& p, int t_base, int mt, const TokTab& tb, int et) {
  for (int j = et; j < mt; j += EPI_THREADS) {
    const int t = t_base + j;
    const bool inj = MODE == GM_INJECT || (MODE == GM_QKV && p.inj_m0 > 0 && t >= p.inj_m0);
    float s = 1.f;
    if (MODE != GM_RESID && MODE != GM_FC) {  // every partial sum of squares at once (H <= 8192: <= 64 parts)
      const bool fold = MODE == GM_QKV && inj;
      const float* src = fold ? p.ss_inj : p.ss_in;
      const int ld = fold ? p.inj_ld : p.ss_ld;
      const int row = fold ? t - p.inj_m0 : t;
      float part[64];
#pragma unroll
      for (int i = 0; i < 64; ++i) part[i] = i < p.ss_parts ? src[(size_t)i * ld + row] : 0.f;
      float acc = 0.f;
#pragma unroll
      for (int i = 0; i < 64; ++i) acc += part[i];
      s = rsqrtf(acc / (float)p.H + p.eps);
    }
    int pos = 0, pg = -1, flag = 0;
    if (MODE == GM_QKV && !inj) {  // block rows: position and page written by the embedding
      const int2 bc = p.bctx[t];
      pos = bc.x;
      pg = bc.y;
      flag = bc.x < p.max_pos ? 1 : 0;  // out-of-range positions were reported by the embedding
    } else if (MODE == GM_QKV || MODE == GM_INJECT) {  // fused-feature rows: the request's slot and position
      int tl = MODE == GM_QKV ? t - p.inj_m0 : t;
      if (MODE == GM_INJECT && p.row_map) tl = p.row_map[tl];  // a compacted row: its request and row
      const int b = tl / p.rows_per_req, ii = tl % p.rows_per_req;
      const int slot = p.slots[b], ne = p.n_eff[b];
      bool live = ii < ne;
      pos = p.pos0[b] + ii;
      if (live && pos >= p.max_pos) {
        dev_error(p.status, DFLASH_DEV_CAPACITY);
        live = false;
      }
      pg = live ? page_of(p, slot, pos) : -1;
      flag = (live ? 1 : 0) | 2;
    }
    tb.s[j] = s;
    tb.pos[j] = pos;
    tb.pg[j] = pg;
    tb.flag[j] = flag;
  }
}

// One warp's EPI_TOK tokens (j0, j0+4, ...) of a chunk: the table's values
// and, for QKV/INJECT, RoPE (cos, sin) of frequencies lane and lane+32 --
// the embedding's per-token rows for block rows, the table at the position
// for fused-feature rows.
struct TokCtx {
  float s[EPI_TOK];
  bool live[EPI_TOK];
  bool inj[EPI_TOK];
  int pos[EPI_TOK], pg[EPI_TOK];
  float2 c0[EPI_TOK], c1[EPI_TOK];
};

template <int MODE>
DFL_DEV void fill_ctx(const GemmParams& p, const TokTab& tb, int tab_t0, int t_first, int j0, int ntok, int lane,
                      TokCtx& c) {
#pragma unroll
  for (int q = 0; q < EPI_TOK; ++q) {
    const int j = j0 + 4 * q;
    const bool ok = j < ntok;  // warp-uniform
    const int k = t_first + (ok ? j : 0) - tab_t0;
    c.s[q] = tb.s[k];
    const int f = ok ? tb.flag[k] : 0;
    c.live[q] = (f & 1) != 0;
    c.inj[q] = (f & 2) != 0;
    c.pos[q] = tb.pos[k];
    c.pg[q] = tb.pg[k];
  }
  if (MODE == GM_QKV || MODE == GM_INJECT) {
    const int D = p.D;
#pragma unroll
    for (int q = 0; q < EPI_TOK; ++q) {
      const bool blk = MODE == GM_QKV && !c.inj[q];
      const float2* row = blk ? p.brope + (size_t)(t_first + j0 + 4 * q) * (D / 2) : p.rope + (size_t)c.pos[q] * (D / 2);
      c.c0[q] = c.live[q] ? row[lane] : make_float2(1.f, 0.f);
      c.c1[q] = (c.live[q] && D == 128) ? row[lane + 32] : make_float2(1.f, 0.f);
    }
  }
}

// Final epilogue for tokens t_first .. t_first+ntok-1 (ntok <= 32) of
// `tile`; staging stg[j][r] holds the fully reduced fp32 accumulators.
// Epilogue warp ew handles tokens j = ew, ew+4, ... (two groups of EPI_TOK
// tokens, ew and ew+16); lane holds rows lane + 32*jj.  The groups run as a
// loop, not unrolled: this code runs cold once per tile, and a second copy
// of it costs more in instruction fetch than the loop does (measured).
// cx holds the contexts of the chunk of cx_key = t_first * 64 + ntok (-1:
// none), both groups' RoPE rows loaded in one round trip: a chunk's contexts
// depend on its tokens only, so every n-tile finalised for the same chunk
// reuses them, and with a single token tile the first chunk's are filled
// while the main loop streams; otherwise they are filled here from the
// shared-memory table tab (its first token tab_t0).  gq/gk: QKV's q/k
// head-norm gains (load_head_gain); hpre (use_hpre, RESID): residual values
// of tokens ew+4q of a single token tile, loaded when the tile started;
// gpre: the tile's gains (RESID/FC).  TIER 0 (one tile of at most 16
// tokens): one token group, its contexts always those filled with the table.
template <int MODE, int TIER>
DFL_DEV void epi_final(const GemmParams& p, int tile, int t_first, int ntok, const float* stg, int ew, int lane,
                       const TokTab& tab, int tab_t0, TokCtx (&cx)[2], int& cx_key, const float* gq, const float* gk,
                       bool use_hpre, const float (&hpre)[EPI_TOK][4], const float (&gpre)[4], int rnd) {
  const int tt_all = tile / p.t_tiles;       // (group, n-tile)
  const int group = tt_all / p.n_tiles;
  const int nt = tt_all % p.n_tiles;
  // FP8 weights: the accumulators carry the rows' scales
  float rs[4] = {1.f, 1.f, 1.f, 1.f};
  if (p.a_fp8) {
    const float* sc = p.a_scale[group] + (size_t)(p.a_tile_off + nt) * 128;
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) rs[jj] = sc[lane + 32 * jj];
  }
  if constexpr (MODE != GM_FC && MODE != GM_RESID && TIER != 0) {
    if (cx_key != t_first * 64 + ntok) {
#pragma unroll
      for (int gi = 0; gi < 2; ++gi)
        if (ew + 16 * gi < ntok) fill_ctx<MODE>(p, tab, tab_t0, t_first, ew + 16 * gi, ntok, lane, cx[gi]);
      cx_key = t_first * 64 + ntok;
    }
  }
#pragma unroll 1
  for (int gi = 0; gi < (TIER == 0 ? 1 : 2); ++gi) {
    const int j0 = ew + 16 * gi;
    if (j0 >= ntok) break;
    bool ok[EPI_TOK];
    int tq[EPI_TOK];
    float x[EPI_TOK][4];
#pragma unroll
    for (int q = 0; q < EPI_TOK; ++q) {
      const int j = j0 + 4 * q;
      ok[q] = j < ntok;  // warp-uniform
      tq[q] = t_first + j;
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) x[q][jj] = ok[q] ? stg[j * 128 + lane + 32 * jj] * rs[jj] : 0.f;
    }

    if constexpr (MODE == GM_RESID || MODE == GM_FC) {
      const int n0 = nt * 128;
      const float(&gn)[4] = gpre;  // the tile's gains, read when the tile started
      float hv[EPI_TOK][4];
      const bool hp = use_hpre && t_first == 0 && gi == 0;
#pragma unroll
      for (int q = 0; q < EPI_TOK; ++q)
#pragma unroll
        for (int jj = 0; jj < 4; ++jj)
          hv[q][jj] = (MODE == GM_RESID && ok[q]) ? (hp ? hpre[q][jj] : p.h[(size_t)tq[q] * p.N + n0 + lane + 32 * jj]) : 0.f;
      float sq[EPI_TOK];
#pragma unroll
      for (int q = 0; q < EPI_TOK; ++q) {
        sq[q] = 0.f;
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          if (MODE == GM_RESID) x[q][jj] += hv[q][jj];
          sq[q] += x[q][jj] * x[q][jj];
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int q = 0; q < EPI_TOK; ++q) sq[q] += __shfl_xor_sync(0xffffffffu, sq[q], o);
#pragma unroll
      for (int q = 0; q < EPI_TOK; ++q) {
        if (!ok[q]) continue;
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const size_t o = (size_t)tq[q] * p.N + n0 + lane + 32 * jj;
          if (MODE == GM_RESID) p.h[o] = x[q][jj];
          p.out[o] = to_f16(x[q][jj] * gn[jj], p.status);
        }
        if (lane == 0) p.ss_out[(size_t)nt * p.M + tq[q]] = sq[q];
      }
    } else {
    TokCtx tcv;
    if constexpr (MODE != GM_RESID && MODE != GM_FC) tcv = gi ? cx[1] : cx[0];
    const TokCtx* tc = &tcv;
    const float* s = tc->s;

    if (MODE == GM_SWIGLU) {
      const int f0 = nt * 64;
#pragma unroll
      for (int q = 0; q < EPI_TOK; ++q) {
        if (!ok[q]) continue;
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
          const float g = x[q][jj] * s[q], u = x[q][jj + 2] * s[q];
          const float a = g / (1.f + __expf(-g)) * u;
          p.out[(size_t)tq[q] * p.N + f0 + lane + 32 * jj] = to_f16(a, p.status);
        }
      }
    } else if (MODE == GM_ARGMAX) {
      const int n0 = nt * 128;
      unsigned long long best[EPI_TOK];
      if (DFL_GEMM_SAMPLING && p.temp_inv > 0.f) {
        // temperature > 0: each drafting row (or, for a target's verify,
        // every row) draws from softmax(logit / T) by the Gumbel-max rule, on
        // its own stream (a separate loop, so the greedy one below keeps its
        // compact code)
        const float tinv = p.temp_inv;
        const bool tgt = p.row0 == 0;
#pragma unroll
        for (int q = 0; q < EPI_TOK; ++q) {
          best[q] = 0ull;
          const int row = tq[q] % DFL_BLOCK;
          const bool smp = ok[q] && (tgt || (row >= 1 && row < p.block));
          unsigned long long skey = 0ull;
          if (smp)
            skey = tgt ? target_stream_key(p.seed, p.slots[tq[q] / DFL_BLOCK], p.bctx[tq[q]].x)
                       : draft_stream_key(p.seed, tq[q] / DFL_BLOCK, rnd, row);
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const int n = n0 + lane + 32 * jj;
            if (ok[q] && n < p.N) {
              const float v = x[q][jj] * s[q];
              if (v != v) {
                dev_error(p.status, DFLASH_DEV_NAN);
                continue;
              }
              if (p.logits) p.logits[(size_t)tq[q] * p.N + n] = v;
              const float sc = smp ? v * tinv + gumbel_at(skey, n) : v;
              const unsigned long long k = argmax_key(sc, (uint32_t)n);
              best[q] = k > best[q] ? k : best[q];
            }
          }
        }
      } else {
#pragma unroll
        for (int q = 0; q < EPI_TOK; ++q) {
          best[q] = 0ull;
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const int n = n0 + lane + 32 * jj;
            if (ok[q] && n < p.N) {
              const float v = x[q][jj] * s[q];
              if (v != v) {
                dev_error(p.status, DFLASH_DEV_NAN);
                continue;
              }
              if (p.logits) p.logits[(size_t)tq[q] * p.N + n] = v;
              const unsigned long long k = argmax_key(v, (uint32_t)n);
              best[q] = k > best[q] ? k : best[q];
            }
          }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int q = 0; q < EPI_TOK; ++q) {
          const unsigned long long other = __shfl_xor_sync(0xffffffffu, best[q], o);
          best[q] = other > best[q] ? other : best[q];
        }
#pragma unroll
      for (int q = 0; q < EPI_TOK; ++q)
        if (ok[q] && lane == 0 && best[q]) atomicMax(p.keys + tq[q], best[q]);
    } else if (MODE == GM_QKV || MODE == GM_INJECT) {
      const int D = p.D;
      int n0, kind, layer;
      float g[4];
      if (MODE == GM_QKV) {
        n0 = nt * 128;
        kind = n0 < p.hq * D ? 0 : (n0 < (p.hq + p.hkv) * D ? 1 : 2);
        layer = p.layer;
#pragma unroll
        for (int j = 0; j < 4; ++j) g[j] = kind == 0 ? gq[j] : gk[j];
      } else {
        n0 = nt * 128 + p.hq * D;  // row index in this layer's wqkv
        kind = n0 < (p.hq + p.hkv) * D ? 1 : 2;
        layer = group;
        if (kind == 1) load_head_gain(p.kn_gain[group], D, lane, g);
      }
      const bool* live = tc->live;
      const bool* inj = tc->inj;
      const int* pos = tc->pos;
      const int* pg = tc->pg;
      const float2* c0 = tc->c0;
      const float2* c1 = tc->c1;
#pragma unroll
      for (int q = 0; q < EPI_TOK; ++q)
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) x[q][jj] *= s[q];
      if (kind < 2) head_norm_rope4(x, g, c0, c1, D, p.eps);
#pragma unroll
      for (int q = 0; q < EPI_TOK; ++q) {
        if (!live[q]) continue;  // warp-uniform
        if (kind == 0 && inj[q]) continue;  // fused-feature rows only append K/V
        const float* xv = x[q];
        if (kind == 0) {
#pragma unroll
          for (int jj = 0; jj < 4; ++jj)
            p.out[(size_t)tq[q] * (p.hq * D) + n0 + lane + 32 * jj] = to_f16(xv[jj], p.status);
          continue;
        }
        if (pg[q] < 0) {  // -2: a padding row of a smaller block
          if (pg[q] == -1) dev_error(p.status, DFLASH_DEV_PAGE);
          continue;
        }
        const int base = (kind == 1 ? p.hq : p.hq + p.hkv) * D;
        f16* pool = kind == 1 ? p.kv.k_pool : p.kv.v_pool;
        const int row = pos[q] & 63;
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int m = n0 + lane + 32 * jj - base;
          const int kh = D == 128 ? m >> 7 : m >> 6, d = m & (D - 1);
          f16* blk = pool + (size_t)layer * p.kv.layer_stride + ((size_t)pg[q] * p.kv.hkv + kh) * (64 * D);
          blk[kind == 1 ? k_swz(row, d) : v_swz(d, row)] = to_f16(xv[jj], p.status);
        }
      }
    }
    }  // not RESID/FC
  }
}

// TIER 2: token tiles of 128+ rows (batched rounds, prefill), shared by a
// cluster, whose split tiles are finalised in several chunks by one CTA;
// only this instance carries the clusters and the pipelined landing of a
// finaliser's next chunk (that code slowed the small-tile instances by ~1 %
// even where it never ran).  TIER 0: one tile of at most 16 tokens (a
// batch-1 round), finalised whole by its last arriving part: no slices.
// TIER 1: the rest.
template <int MODE, bool FP8, int TIER>
__global__ void __launch_bounds__(FP8 ? GEMM_THREADS_FP8 : GEMM_THREADS, 1)
    k_gemm(const __grid_constant__ CUtensorMap tmB, const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* sm = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  const int BN = p.BN;
  const int stages = p.stages;
  const int stage_bytes = A_STAGE_BYTES + BN * 128;
  float* stg = reinterpret_cast<float*>(sm + (size_t)stages * stage_bytes);
  float* red_buf = reinterpret_cast<float*>(sm + (size_t)stages * stage_bytes + STG_BYTES);
  float* tokf = red_buf + (size_t)p.red_items * RED_CHUNK;  // the token table (TOKTAB_BYTES)
  // FP8 weights: each stage's 8 KB block lands here and is converted into the
  // stage's f16 A area by the converter warps
  uint8_t* a8 = sm + (size_t)stages * stage_bytes + STG_BYTES + (size_t)p.red_items * RED_CHUNK * 4 + TOKTAB_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(a8 + (p.a_fp8 ? (size_t)stages * DFL_WBLK8_BYTES : 0));
  uint64_t* empty = full + stages;
  uint64_t* conv = empty + stages;  // FP8: the stage's A converted (the MMA waits on this instead of full)
  uint64_t* tfull = conv + stages;
  uint64_t* tempty = tfull + 2;
  uint64_t* mdone = tempty + 2;
  uint64_t* red = mdone + 1;  // [2] split-K parts landed (one barrier per landing buffer)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(red + 2);
  int* flag = reinterpret_cast<int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t ncols = (uint32_t)p.tmem_cols;
  if (threadIdx.x == 0) trace_at(p, 0, globaltimer());

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, p.cl);  // every cluster CTA's MMAs release the stage
      mbar_init(conv + s, CONV_THREADS);
    }
    mbar_init(tfull + 0, 1);
    mbar_init(tfull + 1, 1);
    mbar_init(tempty + 0, EPI_THREADS);
    mbar_init(tempty + 1, EPI_THREADS);
    mbar_init(mdone, 1);
    mbar_init(red, 1);
    mbar_init(red + 1, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, ncols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // cluster peers write into this CTA's stages and signal its barriers
  if (TIER == 2 && p.cl > 1) cluster_sync_all();
  const uint32_t tmem = *tmem_slot;
  // The QKV projection's dependent, the block attention, reads the page
  // tables and context pages before its own wait: it may launch only once
  // this grid's wait has returned, i.e. once every kernel before it is done.
  if (MODE != GM_QKV) pdl_launch_dependents();
  if (threadIdx.x == 0) trace_at(p, 1, globaltimer());
  // Token rows of this launch: p.M, or the device count p.m_dyn (the live
  // rows of a compacted injection), read after the wait on the kernel that
  // writes it; only the token tiles holding them are scheduled.
  int Mx = p.M, tl = p.t_tiles;
  if (p.m_dyn) {
    pdl_wait();
    const int m = *p.m_dyn;
    Mx = m < 0 ? 0 : (m > p.M ? p.M : m);
    tl = (Mx + BN - 1) / BN;
  }
  const int total_ct = p.groups * p.n_tg * tl;

  // Units (scheduled tile, k-block) are divided over the clusters; the CTAs
  // of a cluster run the same units in lockstep, each on its own n-tile.
  const int KB = p.kblocks;
  const int CL = TIER == 2 ? p.cl : 1;  // clusters share token tiles of 128+ rows only
  const int crank = CL > 1 ? (int)cluster_ctarank() : 0;
  const uint16_t cmask = (uint16_t)((1u << CL) - 1u);
  // Clusters taking part: the grid holds at most one per unit (tile without
  // split) for the launch's rows; with fewer live rows than it was sized
  // for, the clusters past the units present sit out, so every
  // participating cluster has work (split tiles count on every cluster from
  // the first to the last of their units).
  const int c = blockIdx.x / CL;
  int G = gridDim.x / CL;
  const int units_avail = p.allow_split ? total_ct * KB : total_ct;
  if (G > units_avail) G = units_avail;
  int U = total_ct * KB, u0 = 0, u1 = 0;
  if (c < G) {
    if (p.allow_split) {
      u0 = unit_start(c, U, G);
      u1 = unit_start(c + 1, U, G);
    } else {
      u0 = unit_start(c, total_ct, G) * KB;
      u1 = unit_start(c + 1, total_ct, G) * KB;
    }
  }
  bool aborted = false;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    // Tiles of up to 64 tokens with an even ring: lanes 0 and 1 each stream
    // every other stage -- one thread keeps too few bulk copies in flight for
    // full bandwidth (over the GPU ~6.5 TB/s at 16 KB a copy, ~7.2 TB/s from
    // two threads an SM; at 8 KB 3.3 against 6.0).  Per stage a producer only
    // bumps counters and issues two copies; every division happens once per
    // tile.
    const int nprod = (TIER < 2 && DFL_GEMM_PRODUCERS > 1 && (stages & 1) == 0) ? 2 : 1;
    if (lane < nprod) {
      const int pl = lane;  // this producer's units: pl, pl + nprod, ...
      if (pl == 0) prefetch_tmap(&tmB);
      const bool hint = DFL_GEMM_L2_HINT && p.t_tiles == 1;
      const uint64_t pol = policy_evict_first();
      const int KBi = p.kblocks;
      const int n_units = (int)(u1 - u0);
      int tile = (int)(u0 / KB), kb = (int)(u0 % KB), tt = 0;
      const uint8_t* a_ptr = nullptr;
      const int blk_bytes = p.a_fp8 ? DFL_WBLK8_BYTES : A_STAGE_BYTES;
      auto tile_base = [&]() {  // `tile` counts scheduled tiles here
        int rest;
        sched_decode(p, tile, tl, rest, tt);
        const int g = rest / p.n_tg;
        int nt = (rest % p.n_tg) * CL + crank;
        if (nt >= p.n_tiles) nt = p.n_tiles - 1;
        a_ptr = static_cast<const uint8_t*>(p.a[g]) + ((size_t)(p.a_tile_off + nt) * KBi + kb) * blk_bytes;
      };
      tile_base();
      auto advance = [&]() {
        if (++kb == KBi) {
          kb = 0;
          ++tile;
          tile_base();
        } else {
          a_ptr += blk_bytes;
        }
      };
      for (int j = 0; j < pl; ++j) advance();
      auto load_a = [&](int st) {
        uint8_t* dst = p.a_fp8 ? a8 + (size_t)st * DFL_WBLK8_BYTES : sm + (size_t)st * stage_bytes;
        const int CH = blk_bytes / DFL_GEMM_A_CHUNKS;
#pragma unroll
        for (int ch = 0; ch < DFL_GEMM_A_CHUNKS; ++ch) {
          if (hint)
            bulk_load_hint(dst + ch * CH, a_ptr + ch * CH, CH, full + st, pol);
          else
            bulk_load(dst + ch * CH, a_ptr + ch * CH, CH, full + st);
        }
      };
      const uint32_t fill_bytes = (uint32_t)(blk_bytes + BN * 128);  // A (as streamed) + the token tile
      // With a cluster, each CTA loads BN/CL token rows of the tile into every
      // peer's stage (same offsets): the cluster reads each token tile once.
      const int bq = BN / CL;
      auto load_b = [&](int st, int kb_, int tt_) {
        uint8_t* dst = sm + (size_t)st * stage_bytes + A_STAGE_BYTES;
        if (CL > 1)
          tma_load_2d_mc(dst + crank * bq * 128, &tmB, full + st, kb_ * 64, tt_ * BN + crank * bq, cmask);
        else
          tma_load_2d(dst, &tmB, full + st, kb_ * 64, tt_ * BN);
      };
      // Weights do not depend on the previous kernel: fetch the first stages'
      // weight tiles before waiting on it, then the token tiles.
      const int pre = n_units < stages ? n_units : stages;
      int pkb[DFL_GEMM_MAX_STAGES], ptt[DFL_GEMM_MAX_STAGES];
      for (int i = pl; i < pre; i += nprod) {
        mbar_arrive_expect_tx(full + i, fill_bytes);
        load_a(i);
        pkb[i] = kb;
        ptt[i] = tt;
        for (int j = 0; j < nprod; ++j) advance();
      }
      pdl_wait();
      for (int i = pl; i < pre; i += nprod) load_b(i, pkb[i], ptt[i]);
      int issued = pl;  // this producer's next unit
      while (issued < pre) issued += nprod;
      int st = issued % stages;
      uint32_t phase = (uint32_t)((issued / stages) & 1);  // round parity of stage st's next fill
      for (; issued < n_units; issued += nprod) {
        if (!mbar_wait(empty + st, phase ^ 1u, p.status, &aborted)) break;
        mbar_arrive_expect_tx(full + st, fill_bytes);
        load_a(st);
        load_b(st, kb, tt);
        for (int j = 0; j < nprod; ++j) advance();
        st += nprod;
        if (st >= stages) {
          st -= stages;
          phase ^= 1u;
        }
      }
      // drain: every copy this producer issued lands before the CTA may exit
      for (int i = (issued - stages > pl ? issued - stages : pl); i < issued; i += nprod) {
        bool drain_abort = false;
        mbar_wait(full + (i % stages), (uint32_t)((i / stages) & 1), p.status, &drain_abort);
      }
      // and every peer's last release of each stage has arrived here
      if (CL > 1 && !aborted) {
        for (int s2 = 0; s2 < stages && s2 < issued; ++s2) {
          const int last_fill = (issued - 1 - s2) / stages;
          bool drain_abort = false;
          mbar_wait(empty + s2, (uint32_t)(last_fill & 1), p.status, &drain_abort);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    // Tiles of up to 64 tokens: the whole warp runs the loop, converged
    // (every wait's outcome made warp-uniform), and one elected lane issues
    // each MMA and commit -- issued by one lane of an otherwise idle warp, a
    // k-block's wait, fence and four narrow MMAs took about twice as long.
    // Tiles of 128+ tokens are bound by the MMAs themselves: one lane issues
    // (the spinning lanes only cost there), in a loop of its own: the issue
    // rate of one lane's MMAs depends on the exact code around them.
    if constexpr (TIER == 2) {
      if (lane == 0) {
        const uint32_t idesc = idesc_f16_f32(128, BN, p.ab_type);
        int it = 0;
        int seg = 0;
        int s = 0;
        uint32_t phase = 0;
        for (int u = u0; u < u1 && !aborted; ++seg) {
          const int tile = u / KB;
          const int seg_end = (tile + 1) * KB < u1 ? (tile + 1) * KB : u1;
          const int abuf = seg & 1;
          const uint32_t use = (uint32_t)(seg >> 1);
          if (!mbar_wait(tempty + abuf, (use & 1u) ^ 1u, p.status, &aborted)) break;
          tc_fence_after();
          const uint32_t d = tmem + (uint32_t)(abuf * BN);
          for (int k = 0; u < seg_end; ++u, ++k, ++it) {
            if (k > 0 || it > 0) {
              if (++s == stages) {
                s = 0;
                phase ^= 1u;
              }
            }
            if (!mbar_wait((p.a_fp8 ? conv : full) + s, phase, p.status, &aborted)) break;
            if (it == 0) trace_at(p, 2, globaltimer());
            tc_fence_after();
            const uint32_t a_addr = smem_u32(sm + (size_t)s * stage_bytes);
            const uint64_t adesc = sdesc_sw128(a_addr);
            const uint64_t bdesc = sdesc_sw128(a_addr + A_STAGE_BYTES);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              tc_mma_f16(d, adesc + (uint64_t)(2 * kk), bdesc + (uint64_t)(2 * kk), idesc,
                          (k > 0 || kk > 0) ? 1u : 0u);
            if (CL > 1)
              tc_commit_mc(empty + s, cmask);
            else
              tc_commit(empty + s);
          }
          tc_commit(tfull + abuf);
        }
        trace_at(p, 3, globaltimer());
        trace_at(p, 6, (unsigned long long)(u1 - u0) | ((unsigned long long)gridDim.x << 32));
        tc_commit(mdone);
        bool drain_abort = false;
        mbar_wait(mdone, 0, p.status, &drain_abort);
      }
    } else {
      const uint32_t idesc = idesc_f16_f32(128, BN, p.ab_type);
      auto wait_all = [&](uint64_t* bar, uint32_t par) {
        const bool ok = __all_sync(0xffffffffu, mbar_wait(bar, par, p.status, &aborted));
        if (!ok) aborted = true;
        return ok;
      };
      int it = 0;
      int seg = 0;
      int s = 0;
      uint32_t phase = 0;
      for (int u = u0; u < u1 && !aborted; ++seg) {
        const int tile = u / KB;
        const int seg_end = (tile + 1) * KB < u1 ? (tile + 1) * KB : u1;
        const int abuf = seg & 1;
        const uint32_t use = (uint32_t)(seg >> 1);
        if (!wait_all(tempty + abuf, (use & 1u) ^ 1u)) break;
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(abuf * BN);
        for (int k = 0; u < seg_end; ++u, ++k, ++it) {
          if (k > 0 || it > 0) {
            if (++s == stages) {
              s = 0;
              phase ^= 1u;
            }
          }
          if (!wait_all((FP8 ? conv : full) + s, phase)) break;
          if (it == 0 && lane == 0) trace_at(p, 2, globaltimer());
          tc_fence_after();
          const uint32_t a_addr = smem_u32(sm + (size_t)s * stage_bytes);
          const uint64_t adesc = sdesc_sw128(a_addr);
          const uint64_t bdesc = sdesc_sw128(a_addr + A_STAGE_BYTES);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc_mma_f16_elect(d, adesc + (uint64_t)(2 * kk), bdesc + (uint64_t)(2 * kk), idesc,
                             (k > 0 || kk > 0) ? 1u : 0u);
          tc_commit_elect(empty + s);  // one CTA per cluster below 128 tokens
        }
        tc_commit_elect(tfull + abuf);
      }
      if (lane == 0) {
        trace_at(p, 3, globaltimer());
        trace_at(p, 6, (unsigned long long)(u1 - u0) | ((unsigned long long)gridDim.x << 32));
      }
      tc_commit_elect(mdone);
      bool drain_abort = false;
      mbar_wait(mdone, 0, p.status, &drain_abort);
    }
  } else if (warp >= 6) {
    // ------------------------------------------------ FP8 weight converters (warps 6, 7)
    // Each landed 8 KB E4M3 block (row-major, 64 bytes a row) becomes the
    // stage's f16 A operand in the 128-byte-swizzle layout the MMA reads.
    if constexpr (FP8) {
      const int ct = threadIdx.x - GEMM_THREADS;  // 0 .. CONV_THREADS-1
      int s = 0;
      uint32_t phase = 0;
      for (int u = u0, i = 0; u < u1; ++u, ++i) {
        if (i > 0 && ++s == stages) {
          s = 0;
          phase ^= 1u;
        }
        if (!mbar_wait(full + s, phase, p.status, &aborted)) break;
        const uint8_t* src = a8 + (size_t)s * DFL_WBLK8_BYTES;
        uint8_t* dst = sm + (size_t)s * stage_bytes;
        // all of this thread's loads first, then the conversions and stores
        constexpr int NI = 128 * 4 / CONV_THREADS;  // 16-value items per thread
        uint4 v[NI];
#pragma unroll
        for (int k = 0; k < NI; ++k) {
          const int item = ct + k * CONV_THREADS;
          v[k] = *reinterpret_cast<const uint4*>(src + (item >> 2) * 64 + (item & 3) * 16);
        }
#pragma unroll
        for (int k = 0; k < NI; ++k) {
          const int item = ct + k * CONV_THREADS;
          const int row = item >> 2, c8 = item & 3;  // 16 E4M3 values -> two 16-byte f16 chunks
          const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
          uint32_t hv[8];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            hv[2 * j] = e4m3x2_to_f16x2((uint16_t)(w[j] & 0xFFFFu));
            hv[2 * j + 1] = e4m3x2_to_f16x2((uint16_t)(w[j] >> 16));
          }
          uint8_t* drow = dst + row * 128;
          *reinterpret_cast<uint4*>(drow + (((2 * c8) ^ (row & 7)) << 4)) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
          *reinterpret_cast<uint4*>(drow + (((2 * c8 + 1) ^ (row & 7)) << 4)) = make_uint4(hv[4], hv[5], hv[6], hv[7]);
        }
        fence_proxy_async_smem();  // the generic-proxy writes become visible to the MMA's reads
        mbar_arrive(conv + s);
      }
    }
  } else {
    // ------------------------------------------------ epilogue (warps 2..5)
    pdl_wait();
    if (MODE == GM_QKV) pdl_launch_dependents();
    const int q = warp & 3;
    const int r = q * 32 + lane;  // TMEM lane = tile row
    const int et = threadIdx.x - 64;
    const int ew = et >> 5;
    float gq[4], gk[4];
    if (MODE == GM_QKV) {
      load_head_gain(p.qn_gain, p.D, lane, gq);
      load_head_gain(p.kn_gain[0], p.D, lane, gk);
    }
    const int rnd = (MODE == GM_ARGMAX && p.temp_inv > 0.f && p.round) ? *p.round : 0;
    // per-token inputs of the token tile being finalised (not RESID/FC), in
    // shared memory, rebuilt when the token tile changes
    TokTab tab;
    tab.s = tokf;
    tab.pos = reinterpret_cast<int*>(tokf + DFL_BN_MAX);
    tab.pg = tab.pos + DFL_BN_MAX;
    tab.flag = tab.pg + DFL_BN_MAX;
    int tab_tt = -1;
    TokCtx cx[2];  // the contexts of the chunk of cx_key (its first token * 64 + its token count)
    int cx_key = -1;
    // with a single token tile, the contexts of its first 32 tokens (the
    // table's values and their RoPE rows) are filled in registers once, while
    // the main loop streams: the finalisation then issues no load for them
    int seg = 0;
    const int first_tile = u0 / KB;  // this CTA's first segment's scheduled tile
    uint32_t red_phase = 0;  // bit b: the parity of landing barrier red[b]'s next phase
    for (int u = u0; u < u1; ++seg) {
      const int tile_s = u / KB;  // scheduled tile
      const int seg_end = (tile_s + 1) * KB < u1 ? (tile_s + 1) * KB : u1;
      u = seg_end;
      const int abuf = seg & 1;
      const uint32_t use = (uint32_t)(seg >> 1);
      const int tile = tile_of(p, tile_s, crank, tl);
      // RESID/FC: the tile's gains and, with one token tile, the residual
      // inputs of its first 16 tokens, loaded while the accumulators and the
      // split reduction finish
      float hpre[EPI_TOK][4], gpre[4];
      const bool use_hpre = MODE == GM_RESID && p.t_tiles == 1 && tile >= 0;
      if ((MODE == GM_RESID || MODE == GM_FC) && tile >= 0) {
        const int n0 = (int)((tile / p.t_tiles) % p.n_tiles) * 128;
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) gpre[jj] = p.gain[n0 + lane + 32 * jj];
      }
      if (use_hpre) {
        const int n0 = (int)(tile % p.n_tiles) * 128;
#pragma unroll
        for (int q4 = 0; q4 < EPI_TOK; ++q4)
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const int j = ew + 4 * q4;
            hpre[q4][jj] = j < p.M ? p.h[(size_t)j * p.N + n0 + lane + 32 * jj] : 0.f;
          }
      }
      // the token table of this tile's token rows, built while its main loop streams
      if (MODE != GM_RESID && MODE != GM_FC && tile >= 0 && (int)(tile % p.t_tiles) != tab_tt) {
        const int ttb = (int)(tile % p.t_tiles);
        const int tb0 = ttb * BN;
        named_bar_sync(1, EPI_THREADS);  // every thread is done with the previous token tile's table
        const int mtt = (Mx - tb0) < BN ? (Mx - tb0) : BN;
        build_toktab<MODE>(p, tb0, mtt, tab, et);
        named_bar_sync(1, EPI_THREADS);
        tab_tt = ttb;
        cx_key = -1;
        if (p.t_tiles == 1) {  // the first 32-token chunk's contexts, while the main loop streams
          const int n32 = mtt < 32 ? mtt : 32;
#pragma unroll
          for (int gi = 0; gi < 2; ++gi)
            if (ew + 16 * gi < n32) fill_ctx<MODE>(p, tab, tb0, tb0, ew + 16 * gi, n32, lane, cx[gi]);
          cx_key = tb0 * 64 + n32;
        }
      }
      if (!mbar_wait(tfull + abuf, use & 1u, p.status, &aborted)) break;
      tc_fence_after();
      if (tile < 0) {  // a rank past its group's last n-tile
        tc_fence_before();
        mbar_arrive(tempty + abuf);
        continue;
      }
      const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(abuf * BN);
      const int tt = (int)(tile % p.t_tiles);
      const int t_base = tt * BN;
      const int mt = (Mx - t_base) < BN ? (Mx - t_base) : BN;
      int c_first = c, c_last = c;
      if (p.allow_split) {
        c_first = cta_of_unit(tile_s * KB, U, G);
        c_last = cta_of_unit(tile_s * KB + KB - 1, U, G);
      }
      const bool split = c_first != c_last;
      const int nsl = TIER == 0 ? 1 : (mt + 15) >> 4;  // 16-token slices of the tile
      int rank = 0, npar = 1, ct = 16;  // finalisers; tokens per chunk a finaliser takes at once
      if (split) {
        const int my_slot = tile_s == first_tile ? 0 : 1;
        float* w = p.ws + (size_t)((c * CL + crank) * 2 + my_slot) * (DFL_BN_MAX * 128);
        for (int col = 0; col < BN; col += 16) {
          float v[16];
          tmem_ld16(taddr + (uint32_t)col, v);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (col + i < mt) __stcg(w + (size_t)(col + i) * 128 + r, v[i]);
        }
        tc_fence_before();
        mbar_arrive(tempty + abuf);
        named_bar_sync(1, EPI_THREADS);
        // One 16-token slice: the last arriver finalises it at once.  More:
        // the contributors whose unit ranges end in this tile (all but a last
        // one that goes on to the next tile) share the slices, contributor j
        // taking slices j, j+npar, ..., each after a bounded wait for the
        // remaining parts; having no main-loop work left, they hold nothing
        // another CTA waits for.
        const unsigned cnt = (unsigned)(c_last - c_first + 1);
        if (nsl > 1) {
          const int n_end = (int)cnt - (unit_start(c_last + 1, U, G) > (tile_s + 1) * KB ? 1 : 0);
          ct = nsl >= 2 * n_end ? 32 : 16;  // two slices per landing batch when each finaliser has several
          const int nch = (mt + ct - 1) / ct;
          npar = nch < n_end ? nch : n_end;
        }
        if (et == 0) {
          const unsigned old = atomic_add_acq_rel(p.tile_ctr + tile, 1u);
          int go;
          if (nsl == 1) {
            go = old == cnt - 1u ? 0 : -1;
            if (go == 0) p.tile_ctr[tile] = 0;
          } else {
            const int j = c - c_first;
            go = j < npar ? j : -1;
            if (go >= 0 && old != cnt - 1u && !wait_count(p.tile_ctr + tile, cnt, p.status))
              go = -2;  // gave up: skip the slices, still sign off
          }
          *flag = go;
        }
        named_bar_sync(1, EPI_THREADS);
        rank = *flag;
        named_bar_sync(1, EPI_THREADS);
        if (rank == -1) continue;
        if (rank == -2) aborted = true;
      }
      if (split) {
        // The parts' 16-token chunks land in shared memory by bulk copies
        // (one issuing thread, one barrier per batch) and are added in k
        // order by a compact loop -- this code runs cold once per tile.  On
        // the CTA's last segment every weight stage has been consumed, so
        // the whole ring takes a batch; otherwise the p.red_items-chunk buffer.
        // Every part after the first opens its CTA's range (slot 0); the
        // first part is slot 1 unless the tile also opens c_first's.
        const int sl_first = unit_start(c_first, U, G) == tile_s * KB ? 0 : 1;
        const bool ring_free = u == u1;
        float* land = ring_free ? reinterpret_cast<float*>(sm) : red_buf;
        const int cap_items = ring_free ? (stages * stage_bytes) / (RED_CHUNK * 4) : p.red_items;
        const int nparts = c_last - c_first + 1;
        const int nch = (mt + ct - 1) / ct;
        // With room for two chunks' parts (the ring free), the parts of this
        // finaliser's next chunk land while the current one is reduced and
        // run through the epilogue.
        const int half = cap_items / 2;
        const bool pipe = TIER == 2 && DFL_GEMM_LAND_PIPE && ring_free && 2 * nparts <= half && rank + npar < nch;
        auto issue_chunk = [&](int ch, int buf) {  // thread et == 0
          const int tc0 = ch * ct;
          const int subs = (mt - tc0) > 16 && ct == 32 ? 2 : 1;
          const int nitems = nparts * subs;
          float* dst = land + (size_t)buf * half * RED_CHUNK;
          fence_proxy_async_global();  // parts acquired through the tile counter
          mbar_arrive_expect_tx(red + buf, (uint32_t)(nitems * RED_CHUNK * 4));
#pragma unroll 1
          for (int k = 0; k < nitems; ++k) {
            const int sub = k >= nparts ? 1 : 0;
            const int cc = c_first + k - sub * nparts;
            const int sl = cc == c_first ? sl_first : 0;
            bulk_load(dst + k * RED_CHUNK,
                      p.ws + (size_t)((cc * CL + crank) * 2 + sl) * (DFL_BN_MAX * 128) + (size_t)(tc0 + 16 * sub) * 128,
                      RED_CHUNK * 4, red + buf);
          }
        };
        int pbuf = 0;           // pipelined: the buffer of the current chunk
        unsigned in_flight = 0; // pipelined: bit b set while buffer b's copies are issued and not waited for
        if (pipe) {
          if (et == 0) issue_chunk(rank, 0);
          in_flight = 1u;
        }
        for (int ch = rank; ch < nch && !aborted; ch += npar) {
          const int tc0 = ch * ct;
          const int subs = TIER != 0 && (mt - tc0) > 16 && ct == 32 ? 2 : 1;  // 16-token slices in this chunk
          float v0[16], v1[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) v0[i] = v1[i] = 0.f;
          const int nitems = nparts * subs;  // (sub, part), part fastest
          if (pipe) {
            if (ch + npar < nch) {
              if (et == 0) issue_chunk(ch + npar, pbuf ^ 1);
              in_flight |= 1u << (pbuf ^ 1);
            }
            if (!mbar_wait(red + pbuf, (red_phase >> pbuf) & 1u, p.status, &aborted)) break;
            red_phase ^= 1u << pbuf;
            in_flight &= ~(1u << pbuf);
            const float* lb = land + (size_t)pbuf * half * RED_CHUNK + r;
#pragma unroll 1
            for (int k = 0; k < nitems; ++k) {
              const float* src = lb + k * RED_CHUNK;
              if (k < nparts) {
#pragma unroll
                for (int i = 0; i < 16; ++i) v0[i] += src[i * 128];
              } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) v1[i] += src[i * 128];
              }
            }
          } else {
            for (int it0 = 0; it0 < nitems && !aborted; it0 += cap_items) {
              const int nb = (nitems - it0) < cap_items ? (nitems - it0) : cap_items;
              if (et == 0) {
                fence_proxy_async_global();  // parts acquired through the tile counter
                mbar_arrive_expect_tx(red, (uint32_t)(nb * RED_CHUNK * 4));
#pragma unroll 1
                for (int k = 0; k < nb; ++k) {
                  const int item = it0 + k;
                  const int sub = item >= nparts ? 1 : 0;
                  const int cc = c_first + item - sub * nparts;
                  const int sl = cc == c_first ? sl_first : 0;
                  bulk_load(land + k * RED_CHUNK,
                            p.ws + (size_t)((cc * CL + crank) * 2 + sl) * (DFL_BN_MAX * 128) + (size_t)(tc0 + 16 * sub) * 128,
                            RED_CHUNK * 4, red);
                }
              }
              if (!mbar_wait(red, red_phase & 1u, p.status, &aborted)) break;
              red_phase ^= 1u;
#pragma unroll 1
              for (int k = 0; k < nb; ++k) {
                const float* src = land + k * RED_CHUNK + r;
                if (it0 + k < nparts) {
#pragma unroll
                  for (int i = 0; i < 16; ++i) v0[i] += src[i * 128];
                } else {
#pragma unroll
                  for (int i = 0; i < 16; ++i) v1[i] += src[i * 128];
                }
              }
              named_bar_sync(1, EPI_THREADS);  // landing area free for the next batch
            }
          }
#pragma unroll
          for (int i = 0; i < 16; ++i) stg[i * 128 + r] = v0[i];
          if (subs == 2) {
#pragma unroll
            for (int i = 0; i < 16; ++i) stg[(16 + i) * 128 + r] = v1[i];
          }
          named_bar_sync(1, EPI_THREADS);
          epi_final<MODE, TIER>(p, (int)tile, t_base + tc0, (mt - tc0) < ct ? (mt - tc0) : ct, stg, ew, lane, tab,
                          t_base, cx, cx_key, gq, gk, use_hpre, hpre, gpre, rnd);
          named_bar_sync(1, EPI_THREADS);  // staging (and, pipelined, this chunk's landing buffer) free
          pbuf ^= 1;
        }
        // gave up while copies were in flight: they land before the CTA moves on
        for (int b = 0; b < 2; ++b)
          if (in_flight & (1u << b)) {
            bool drain_abort = false;
            mbar_wait(red + b, (red_phase >> b) & 1u, p.status, &drain_abort);
          }
        // several slices: the last finaliser to finish clears the tile's counters
        if (nsl > 1 && et == 0) {
          if (atomicAdd(p.tile_fin + tile, 1u) == (unsigned)(npar - 1)) {
            p.tile_ctr[tile] = 0;
            p.tile_fin[tile] = 0;
          }
        }
      } else {
        for (int tc0 = 0; tc0 < mt; tc0 += 32) {
          float v0[16], v1[16];
          const bool two = TIER != 0 && tc0 + 16 < BN;  // a second 16-column chunk in this 32-token chunk
          tmem_ld16(taddr + (uint32_t)tc0, v0);
          if (two) tmem_ld16(taddr + (uint32_t)(tc0 + 16), v1);
#pragma unroll
          for (int i = 0; i < 16; ++i) stg[i * 128 + r] = v0[i];
          if (two) {
#pragma unroll
            for (int i = 0; i < 16; ++i) stg[(16 + i) * 128 + r] = v1[i];
          }
          named_bar_sync(1, EPI_THREADS);
          epi_final<MODE, TIER>(p, (int)tile, t_base + tc0, (mt - tc0) < 32 ? (mt - tc0) : 32, stg, ew, lane, tab,
                          t_base, cx, cx_key, gq, gk, use_hpre, hpre, gpre, rnd);
          named_bar_sync(1, EPI_THREADS);
        }
      }
      if (!split) {
        tc_fence_before();
        mbar_arrive(tempty + abuf);
      }
    }
    if (threadIdx.x == 64) trace_at(p, 4, globaltimer());
  }

  __syncthreads();
  // no CTA leaves while a peer may still write into it or signal its barriers
  if (TIER == 2 && p.cl > 1) cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, ncols);
  }
  if (threadIdx.x == 0) {
    uint32_t smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    trace_at(p, 7, smid);
    trace_at(p, 5, globaltimer());
  }
  if (MODE == GM_ARGMAX) {
    // The last CTA to finish turns the per-token argmax keys of block rows
    // 1..S-1 into draft ids and clears the keys for the next round.
    int* done_flag = flag + 1;
    if (threadIdx.x == 0) {
      __threadfence();
      const unsigned old = atomicAdd(p.done_ctr, 1u);
      *done_flag = old == gridDim.x - 1;
    }
    __syncthreads();
    if (*done_flag) {
      __threadfence();
      const int batch = p.M / DFL_BLOCK;
      const int nd = p.block - p.row0;  // tokens per request: block rows row0..S-1
      for (int idx = threadIdx.x; idx < batch * nd; idx += blockDim.x) {
        const int b = idx / nd, i = idx % nd + p.row0;
        const unsigned long long k = __ldcg(p.keys + b * DFL_BLOCK + i);
        p.draft[idx] = k ? (int)argmax_key_index(k) : 0;
      }
      __syncthreads();
      for (int idx = threadIdx.x; idx < p.M; idx += blockDim.x) p.keys[idx] = 0ull;
      if (threadIdx.x == 0) *p.done_ctr = 0u;
    }
  }
}

}  // namespace

// Split-K part chunks (8 KB) the reduction lands at once while the ring is
// still in use: whatever shared memory the ring leaves, 4 to 16.
int gemm_red_items(int BN, int stages, int fp8) {
  const long long left = 232448LL - 1024 - (long long)stages * (A_STAGE_BYTES + BN * 128 + (fp8 ? DFL_WBLK8_BYTES : 0)) -
                         STG_BYTES - TOKTAB_BYTES - 512;
  const long long n = left / (RED_CHUNK * 4);
  return (int)(n < RED_PARTS ? RED_PARTS : (n > DFL_GEMM_RED_MAX ? DFL_GEMM_RED_MAX : n));
}

size_t gemm_smem_bytes(int BN, int stages, int fp8) {
  return 1024 + (size_t)stages * (A_STAGE_BYTES + BN * 128 + (fp8 ? DFL_WBLK8_BYTES : 0)) + STG_BYTES +
         (size_t)gemm_red_items(BN, stages, fp8) * RED_CHUNK * 4 + TOKTAB_BYTES + (size_t)(3 * stages + 7) * 8 + 16;
}

// Weight-ring depth.  Six 16 KB stages per SM already keep HBM streaming at
// full rate; deeper rings only lengthen the queues that the split-K
// reduction's L2 round trips wait behind (measured: the Qwen3-8B-shaped round
// is fastest at 6-7 stages, 2.5% slower at 12).  The lm_head, one long
// stream with short tails, runs best at 8.
int gemm_pick_stages(int BN, int mode, int fp8) {
  const size_t budget = 232448 - 1024 - STG_BYTES - RED_BYTES - TOKTAB_BYTES - 512;
  int st = (int)(budget / (size_t)(A_STAGE_BYTES + BN * 128 + (fp8 ? DFL_WBLK8_BYTES : 0)));
  const int cap = mode == GM_ARGMAX ? 8 : 6;
  st = st > cap ? cap : st;
  return st > DFL_GEMM_MAX_STAGES ? DFL_GEMM_MAX_STAGES : st;
}

template <int MODE, bool FP8>
cudaError_t set_smem_attr(int tier) {
  const cudaFuncAttribute A = cudaFuncAttributeMaxDynamicSharedMemorySize;
  return tier == 2   ? cudaFuncSetAttribute(k_gemm<MODE, FP8, 2>, A, 232448)
         : tier == 1 ? cudaFuncSetAttribute(k_gemm<MODE, FP8, 1>, A, 232448)
                     : cudaFuncSetAttribute(k_gemm<MODE, FP8, 0>, A, 232448);
}

template <int MODE, bool FP8>
cudaError_t launch_inst(cudaLaunchConfig_t* cfg, const CUtensorMap& B, const GemmParams& p) {
  if (p.BN >= 128) return cudaLaunchKernelEx(cfg, k_gemm<MODE, FP8, 2>, B, p);
  if (p.M <= 16 && p.t_tiles == 1 && !p.m_dyn) return cudaLaunchKernelEx(cfg, k_gemm<MODE, FP8, 0>, B, p);
  return cudaLaunchKernelEx(cfg, k_gemm<MODE, FP8, 1>, B, p);
}

cudaError_t gemm_init_attributes() {
  cudaError_t e;
  for (int big = 0; big < 3; ++big) {
    if ((e = set_smem_attr<GM_QKV, false>(big))) return e;
    if ((e = set_smem_attr<GM_INJECT, false>(big))) return e;
    if ((e = set_smem_attr<GM_RESID, false>(big))) return e;
    if ((e = set_smem_attr<GM_SWIGLU, false>(big))) return e;
    if ((e = set_smem_attr<GM_FC, false>(big))) return e;
    if ((e = set_smem_attr<GM_ARGMAX, false>(big))) return e;
    if ((e = set_smem_attr<GM_QKV, true>(big))) return e;
    if ((e = set_smem_attr<GM_INJECT, true>(big))) return e;
    if ((e = set_smem_attr<GM_RESID, true>(big))) return e;
    if ((e = set_smem_attr<GM_SWIGLU, true>(big))) return e;
    if ((e = set_smem_attr<GM_ARGMAX, true>(big))) return e;
  }
  return cudaSuccess;
}

int gemm_max_clusters(int BN, int stages, int cl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(cl * 64));
  cfg.blockDim = dim3(GEMM_THREADS);
  cfg.dynamicSmemBytes = gemm_smem_bytes(BN, stages, 0);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, k_gemm<GM_ARGMAX, false, 2>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

cudaError_t gemm_launch(const CUtensorMap& B, const GemmParams& p, int grid, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(p.a_fp8 ? GEMM_THREADS_FP8 : GEMM_THREADS);  // converter warps for FP8 weights only
  cfg.dynamicSmemBytes = gemm_smem_bytes(p.BN, p.stages, p.a_fp8);
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if (p.cl > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = (unsigned)p.cl;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = (unsigned)na;
  switch (p.mode) {
    case GM_QKV: return p.a_fp8 ? launch_inst<GM_QKV, true>(&cfg, B, p) : launch_inst<GM_QKV, false>(&cfg, B, p);
    case GM_INJECT: return p.a_fp8 ? launch_inst<GM_INJECT, true>(&cfg, B, p) : launch_inst<GM_INJECT, false>(&cfg, B, p);
    case GM_RESID: return p.a_fp8 ? launch_inst<GM_RESID, true>(&cfg, B, p) : launch_inst<GM_RESID, false>(&cfg, B, p);
    case GM_SWIGLU: return p.a_fp8 ? launch_inst<GM_SWIGLU, true>(&cfg, B, p) : launch_inst<GM_SWIGLU, false>(&cfg, B, p);
    case GM_FC: return launch_inst<GM_FC, false>(&cfg, B, p);  // the fusion projection stays bf16
    case GM_ARGMAX: return p.a_fp8 ? launch_inst<GM_ARGMAX, true>(&cfg, B, p) : launch_inst<GM_ARGMAX, false>(&cfg, B, p);
  }
  return cudaErrorInvalidValue;
}
