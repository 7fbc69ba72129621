// Block attention: the 16 block queries of every query head attend, with no
// mask, to [context K/V ; block K/V] of their KV head (grouped-query attention).
//
// Grid (split, kv_head, request).  One CTA owns the G = hq/hkv query heads of
// one KV head (16 block rows each) and a contiguous range of the request's
// 64-position pages.  Each page of K (64 x D) and V^T (D x 64) is a
// contiguous 2 x 8..16 KB block stored pre-swizzled in HBM, so an untiled TMA
// bulk copy lands it in shared memory already in a bank-conflict-free layout
// for ldmatrix.  Q.K^T and P.V run on warp MMAs (m16n8k16, f16 in, fp32
// accumulate), the softmax is online in the log2 domain with quad shuffles.
// The splits of one (request, KV head) are one thread-block cluster; their
// fp32 partials (O, running max, running sum) stay in shared memory and are
// merged in split order over distributed shared memory -- deterministic, no
// global scratch.
#include "common.cuh"
#include "internal.h"

namespace {

// Splits of one (request, KV head) are one thread-block cluster: up to 16
// CTAs (a non-portable cluster size, used only where the GPU can hold the
// clusters at once; see attn_max_active_clusters).
constexpr int ATTN_MAX_SPLITS = 16;

template <int D>
struct AttnCfg {
#ifndef DFL_ATTN_STAGES
#define DFL_ATTN_STAGES 6
#endif
  static constexpr int STAGES = D == 128 ? DFL_ATTN_STAGES : 8;  // pages in flight per CTA
  static constexpr int BLK_BYTES = 64 * D * 2;               // one K (or V) page block
  static constexpr int STAGE_BYTES = 2 * BLK_BYTES;
  static constexpr int MAX_PIDS = 512;                       // page ids prefetched to shared memory
  static constexpr int SMEM = STAGES * STAGE_BYTES + 128 + MAX_PIDS * 4;  // + barriers, page ids
};

// Timeline stamps (p.trace non-null), per CTA in grid order: 0 entry, 1 context
// length known, 2 first page landed, 3 pages done, 4 partial published, 5 exit;
// with the entry, 6 = the launch's CTA count in the high 32 bits (low bits 0).
DFL_DEV void atrace(const AttnParams& p, int ev) {
  if (p.trace) {
    const size_t cta = ((size_t)blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
    p.trace[cta * 8 + ev] = globaltimer();
    if (ev == 0) p.trace[cta * 8 + 6] = (unsigned long long)gridDim.x * gridDim.y * gridDim.z << 32;
  }
}

// The QKV projection before this kernel lets it launch only after that
// projection's own dependency wait, so every earlier kernel (page
// allocation, injection, embedding) is complete when this one starts: with
// p.early the slot, its length, its page table and the pages holding no
// block row are read at once, and the block's own K/V and its queries,
// written by the projection, only after this kernel's wait.  A folded round
// (the projection also appends the new context rows) clears p.early.

// A split's partial (nf floats from shared memory) to its global slot.
DFL_DEV void copy_partial(const AttnParams& p, const float* part, int nf, int slot, int D) {
  float* dst = p.part + (size_t)slot * attn_part_floats(D);
  for (int i = 4 * (int)threadIdx.x; i < nf; i += 4 * (int)blockDim.x)
    *reinterpret_cast<float4*>(dst + i) = *reinterpret_cast<const float4*>(part + i);
}

// Combines the splits' partials of each (request, KV head): one CTA per 16
// rows (one query head's block tokens), 16 threads per row, each taking D/16
// output columns.  Every split's max and sum and the first 16 splits'
// unnormalised outputs are loaded at once (one round trip), any further
// splits' outputs in groups of 16, and summed in split order.
constexpr int MERGE_TPR = 16;      // threads per row
constexpr int MERGE_MAX_SPLITS = 32;
constexpr int MERGE_GROUP = 16;    // splits whose outputs are loaded at once

template <int D>
__global__ void __launch_bounds__(16 * MERGE_TPR) k_attn_merge(const AttnParams p) {
  constexpr int PS = D + 4;
  constexpr int PF = attn_part_floats(D);
  constexpr int DC = D / MERGE_TPR;  // columns per thread (8 or 4)
  constexpr int NV = DC / 4;         // float4 per split
  pdl_launch_dependents();
  pdl_wait();
  const int pair = blockIdx.x;
  const int b = pair / p.hkv, kvh = pair % p.hkv;
  const int G = p.hq / p.hkv, rows = G * 16;
  const int r = blockIdx.y * 16 + ((int)threadIdx.x / MERGE_TPR);
  const int d0 = ((int)threadIdx.x % MERGE_TPR) * DC;
  if (r >= rows) return;
  const int nsp = p.n_splits;
  const float* base = p.part + (size_t)pair * nsp * PF;
  float mv[MERGE_MAX_SPLITS], lv[MERGE_MAX_SPLITS];
  float4 v0[MERGE_GROUP][NV];  // the first group's outputs, loaded with the maxima and sums
#pragma unroll
  for (int sp = 0; sp < MERGE_MAX_SPLITS; ++sp) {
    mv[sp] = -INFINITY;
    lv[sp] = 0.f;
    if (sp < nsp) {
      lv[sp] = base[(size_t)sp * PF + rows * PS + rows + r];
      mv[sp] = base[(size_t)sp * PF + rows * PS + r];
    }
  }
#pragma unroll
  for (int k = 0; k < MERGE_GROUP; ++k)
#pragma unroll
    for (int c4 = 0; c4 < NV; ++c4)
      v0[k][c4] = k < nsp ? *reinterpret_cast<const float4*>(base + (size_t)k * PF + r * PS + d0 + 4 * c4)
                          : make_float4(0.f, 0.f, 0.f, 0.f);
  float M = -INFINITY;
#pragma unroll
  for (int sp = 0; sp < MERGE_MAX_SPLITS; ++sp)
    if (lv[sp] > 0.f) M = fmaxf(M, mv[sp]);
  float L = 0.f;
#pragma unroll
  for (int sp = 0; sp < MERGE_MAX_SPLITS; ++sp) {
    const float w = lv[sp] > 0.f ? exp2f(mv[sp] - M) : 0.f;
    mv[sp] = w;  // now the split's weight
    L += w * lv[sp];
  }
  float acc[DC];
#pragma unroll
  for (int c = 0; c < DC; ++c) acc[c] = 0.f;
#pragma unroll
  for (int g = 0; g < MERGE_MAX_SPLITS; g += MERGE_GROUP) {
    if (g >= nsp) break;
    float4 v[MERGE_GROUP][NV];
#pragma unroll
    for (int k = 0; k < MERGE_GROUP; ++k)
#pragma unroll
      for (int c4 = 0; c4 < NV; ++c4)
        v[k][c4] = g == 0 ? v0[k][c4]
                          : (g + k < nsp ? *reinterpret_cast<const float4*>(base + (size_t)(g + k) * PF + r * PS + d0 + 4 * c4)
                                         : make_float4(0.f, 0.f, 0.f, 0.f));
#pragma unroll
    for (int k = 0; k < MERGE_GROUP; ++k) {
      const float w = mv[g + k];  // 0 past the last split
#pragma unroll
      for (int c4 = 0; c4 < NV; ++c4) {
        acc[4 * c4] += w * v[k][c4].x;
        acc[4 * c4 + 1] += w * v[k][c4].y;
        acc[4 * c4 + 2] += w * v[k][c4].z;
        acc[4 * c4 + 3] += w * v[k][c4].w;
      }
    }
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  const int h = r / 16, t = r % 16;
  f16* dst = p.out + ((size_t)(b * DFL_BLOCK + t) * p.hq + kvh * G + h) * D + d0;
#pragma unroll
  for (int c = 0; c < DC; c += 4)
    *reinterpret_cast<uint2*>(dst + c) =
        make_uint2(pack_f16x2(acc[c] * inv, acc[c + 1] * inv), pack_f16x2(acc[c + 2] * inv, acc[c + 3] * inv));
}

template <int D, int G, int KS>
__global__ void __launch_bounds__(G * KS * 32) k_attn(const AttnParams p) {
  using C = AttnCfg<D>;
  constexpr int KPW = 64 / KS;   // keys of a page per warp
  constexpr int NKG = KPW / 16;  // 16-key groups per warp
  constexpr int PS = D + 4;      // padded row stride (floats) of a partial
  extern __shared__ __align__(128) uint8_t sm[];
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + C::STAGES * C::STAGE_BYTES);
  int* pids = reinterpret_cast<int*>(sm + C::STAGES * C::STAGE_BYTES + 128);

  const int split = blockIdx.x, kvh = blockIdx.y, b = p.order ? p.order[blockIdx.z] : (int)blockIdx.z;
  const int head0 = kvh * G;  // first query head
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hw = warp % G;    // query head of this warp within the group
  const int half = warp / G;  // which KPW keys of every page
  const int g = lane >> 2, c4 = lane & 3;
  const int rows = G * 16;
  const int hq = p.hq, hkv = p.hkv;

  if (threadIdx.x == 0) {
    atrace(p, 0);
    for (int s = 0; s < C::STAGES; ++s) mbar_init(full + s, 1);
    fence_mbar_init();
  }
  pdl_launch_dependents();
  if (!p.early) pdl_wait();

  const int slot = p.slots[b];
  const int nv = p.n_valid ? min(max(p.n_valid[b], 1), DFL_BLOCK) : p.block;  // live block rows
  const int nkeys = p.ctx_len[slot] + nv;             // context + live block rows
  const int npages = (nkeys + 63) >> 6;
  const int pb = (int)((long long)split * npages / p.n_splits);  // balanced page ranges
  const int pe = (int)((long long)(split + 1) * npages / p.n_splits);
  const int ctx_pages = (nkeys - nv) >> 6;            // pages holding no block row
  // keys of rows g and g+8: all, or (causal) the context and block rows up to
  // the row itself (padding rows: up to the last live row)
  const int lim0 = p.causal ? nkeys - nv + min(g, nv - 1) + 1 : nkeys;
  const int lim1 = p.causal ? nkeys - nv + min(g + 8, nv - 1) + 1 : nkeys;
  const f16* kbase = p.kv.k_pool + (size_t)p.layer * p.kv.layer_stride;
  const f16* vbase = p.kv.v_pool + (size_t)p.layer * p.kv.layer_stride;
  const int* pt = p.kv.page_table + (size_t)slot * p.kv.max_pages_per_slot;
  // this CTA's page ids, read in parallel once (not one dependent load per copy)
  for (int i = threadIdx.x; i < pe - pb && i < C::MAX_PIDS; i += blockDim.x)
    pids[i] = pb + i < p.kv.max_pages_per_slot ? pt[pb + i] : -1;
  __syncthreads();
  if (threadIdx.x == 0) atrace(p, 1);

  auto issue = [&](int s, int page_idx) {
    const int li = page_idx - pb;
    int pg = li < C::MAX_PIDS ? pids[li] : (page_idx < p.kv.max_pages_per_slot ? pt[page_idx] : -1);
    if (pg < 0 || pg >= p.kv.max_pages) {
      dev_error(p.status, DFLASH_DEV_PAGE);
      pg = 0;
    }
    const size_t off = ((size_t)pg * hkv + kvh) * (64 * D);
    uint8_t* dst = sm + s * C::STAGE_BYTES;
    mbar_arrive_expect_tx(full + s, C::STAGE_BYTES);
    bulk_load(dst, kbase + off, C::BLK_BYTES, full + s);
    bulk_load(dst + C::BLK_BYTES, vbase + off, C::BLK_BYTES, full + s);
  };
  int issued = 0;  // meaningful in thread 0 only
  if (p.early) {
    if (threadIdx.x == 0)  // context pages first, then (after the wait) the block's
      for (; issued < C::STAGES && pb + issued < pe && pb + issued < ctx_pages; ++issued) issue(issued, pb + issued);
    pdl_wait();
  }
  if (threadIdx.x == 0)
    for (; issued < C::STAGES && pb + issued < pe; ++issued) issue(issued, pb + issued);

  // Q fragments of this warp's query head (16 block rows x D) in registers.
  const int j = head0 + hw;
  uint32_t qa[D / 16][4];
  {
    const f16* q0 = p.q + ((size_t)(b * DFL_BLOCK) * hq + j) * D;
    const size_t rs = (size_t)hq * D;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const int col = kk * 16 + 2 * c4;
      qa[kk][0] = *reinterpret_cast<const uint32_t*>(q0 + g * rs + col);
      qa[kk][1] = *reinterpret_cast<const uint32_t*>(q0 + (g + 8) * rs + col);
      qa[kk][2] = *reinterpret_cast<const uint32_t*>(q0 + g * rs + col + 8);
      qa[kk][3] = *reinterpret_cast<const uint32_t*>(q0 + (g + 8) * rs + col + 8);
    }
  }

  float o[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  bool aborted = false;
  const int mi = lane >> 3, rr = lane & 7;

  int it = 0;
  for (int pi = pb; pi < pe; ++pi, ++it) {
    const int s = it % C::STAGES;
    const bool ok = mbar_wait(full + s, (uint32_t)((it / C::STAGES) & 1), p.status, &aborted);
    if (it == 0 && threadIdx.x == 0) atrace(p, 2);
    if (ok) {
      const int valid0 = min(64, lim0 - pi * 64), valid1 = min(64, lim1 - pi * 64);
      const uint32_t kb_addr = smem_u32(sm + s * C::STAGE_BYTES);
      const uint32_t vb_addr = kb_addr + C::BLK_BYTES;
      float sc[2 * NKG][4];
#pragma unroll
      for (int i = 0; i < 2 * NKG; ++i) sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.f;
      // S = Q K^T over this warp's keys of the page
#pragma unroll
      for (int kg = 0; kg < NKG; ++kg) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const int key = half * KPW + kg * 16 + (mi >> 1) * 8 + rr;
          const int chunk = kk * 2 + (mi & 1);
          const uint32_t addr =
              kb_addr + 2u * (uint32_t)((chunk >> 3) * (64 * 64) + key * 64 + (((chunk & 7) ^ (key & 7)) << 3));
          uint32_t b0, b1, b2, b3;
          ldsm_x4(addr, b0, b1, b2, b3);
          mma_f16_16816(sc[2 * kg], qa[kk], b0, b1);
          mma_f16_16816(sc[2 * kg + 1], qa[kk], b2, b3);
        }
      }
      // online softmax (log2 domain), rows g and g+8 of this warp; a row
      // whose keys so far are all masked keeps max -inf and contributes 0
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 2 * NKG; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int key = half * KPW + nt * 8 + 2 * c4 + (e & 1);
          float v = sc[nt][e] * p.scale_log2;
          if (key >= (e < 2 ? valid0 : valid1)) v = -INFINITY;
          sc[nt][e] = v;
        }
        mx0 = fmaxf(mx0, fmaxf(sc[nt][0], sc[nt][1]));
        mx1 = fmaxf(mx1, fmaxf(sc[nt][2], sc[nt][3]));
      }
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const float ref0 = mn0 == -INFINITY ? 0.f : mn0, ref1 = mn1 == -INFINITY ? 0.f : mn1;
      const float a0 = exp2f(m0 - ref0), a1 = exp2f(m1 - ref1);
      float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
      for (int nt = 0; nt < 2 * NKG; ++nt) {
        sc[nt][0] = exp2f(sc[nt][0] - ref0);
        sc[nt][1] = exp2f(sc[nt][1] - ref0);
        sc[nt][2] = exp2f(sc[nt][2] - ref1);
        sc[nt][3] = exp2f(sc[nt][3] - ref1);
        rs0 += sc[nt][0] + sc[nt][1];
        rs1 += sc[nt][2] + sc[nt][3];
      }
      l0 = l0 * a0 + rs0;
      l1 = l1 * a1 + rs1;
      m0 = mn0;
      m1 = mn1;
#pragma unroll
      for (int nd = 0; nd < D / 8; ++nd) {
        o[nd][0] *= a0;
        o[nd][1] *= a0;
        o[nd][2] *= a1;
        o[nd][3] *= a1;
      }
      // O += P V  (V^T page: rows = dims, 64 keys per row)
#pragma unroll
      for (int k2 = 0; k2 < NKG; ++k2) {
        uint32_t pa[4];
        pa[0] = pack_f16x2(sc[2 * k2][0], sc[2 * k2][1]);
        pa[1] = pack_f16x2(sc[2 * k2][2], sc[2 * k2][3]);
        pa[2] = pack_f16x2(sc[2 * k2 + 1][0], sc[2 * k2 + 1][1]);
        pa[3] = pack_f16x2(sc[2 * k2 + 1][2], sc[2 * k2 + 1][3]);
#pragma unroll
        for (int nd = 0; nd < D / 8; nd += 2) {
          const int dim = (nd + (mi >> 1)) * 8 + rr;
          const int chunk = 2 * (half * NKG + k2) + (mi & 1);
          const uint32_t addr = vb_addr + 2u * (uint32_t)(dim * 64 + ((chunk ^ (dim & 7)) << 3));
          uint32_t b0, b1, b2, b3;
          ldsm_x4(addr, b0, b1, b2, b3);
          mma_f16_16816(o[nd], pa, b0, b1);
          mma_f16_16816(o[nd + 1], pa, b2, b3);
        }
      }
    }
    __syncthreads();
    if (threadIdx.x == 0 && !aborted && pi + C::STAGES < pe) {
      issue(s, pi + C::STAGES);
      ++issued;
    }
  }
  if (threadIdx.x == 0 && aborted) {
    // let copies already in flight land before the CTA exits
    for (int i = (issued > C::STAGES ? issued - C::STAGES : 0); i < issued; ++i) {
      bool drain_abort = false;
      mbar_wait(full + (i % C::STAGES), (uint32_t)((i / C::STAGES) & 1), p.status, &drain_abort);
    }
  }

  if (threadIdx.x == 0) atrace(p, 3);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  const int r0 = hw * 16 + g, r1 = r0 + 8;

  // partial layout in shared memory: [rows][PS] unnormalised O, then the
  // running max [rows] and running sum [rows]
  float* part = reinterpret_cast<float*>(sm);
  if (KS == 2) {
    // the second key half of every head hands its state to the first
    constexpr int PART_FLOATS = G * 16 * PS + 2 * G * 16;
    float* xch = part + ((PART_FLOATS + 31) & ~31);
    __syncthreads();  // every warp is past its last read of the page stages
    if (half == 1) {
#pragma unroll
      for (int nd = 0; nd < D / 8; ++nd) {
        const int d = nd * 8 + 2 * c4;
        *reinterpret_cast<float2*>(xch + r0 * PS + d) = make_float2(o[nd][0], o[nd][1]);
        *reinterpret_cast<float2*>(xch + r1 * PS + d) = make_float2(o[nd][2], o[nd][3]);
      }
      if (c4 == 0) {
        xch[rows * PS + r0] = m0;
        xch[rows * PS + r1] = m1;
        xch[rows * PS + rows + r0] = l0;
        xch[rows * PS + rows + r1] = l1;
      }
    }
    __syncthreads();
    if (half == 0) {
      const float mb0 = xch[rows * PS + r0], mb1 = xch[rows * PS + r1];
      const float lb0 = xch[rows * PS + rows + r0], lb1 = xch[rows * PS + rows + r1];
      const float M0 = fmaxf(l0 > 0.f ? m0 : -INFINITY, lb0 > 0.f ? mb0 : -INFINITY);
      const float M1 = fmaxf(l1 > 0.f ? m1 : -INFINITY, lb1 > 0.f ? mb1 : -INFINITY);
      const float wa0 = l0 > 0.f ? exp2f(m0 - M0) : 0.f, wb0 = lb0 > 0.f ? exp2f(mb0 - M0) : 0.f;
      const float wa1 = l1 > 0.f ? exp2f(m1 - M1) : 0.f, wb1 = lb1 > 0.f ? exp2f(mb1 - M1) : 0.f;
#pragma unroll
      for (int nd = 0; nd < D / 8; ++nd) {
        const int d = nd * 8 + 2 * c4;
        const float2 x0 = *reinterpret_cast<const float2*>(xch + r0 * PS + d);
        const float2 x1 = *reinterpret_cast<const float2*>(xch + r1 * PS + d);
        o[nd][0] = o[nd][0] * wa0 + x0.x * wb0;
        o[nd][1] = o[nd][1] * wa0 + x0.y * wb0;
        o[nd][2] = o[nd][2] * wa1 + x1.x * wb1;
        o[nd][3] = o[nd][3] * wa1 + x1.y * wb1;
      }
      l0 = l0 * wa0 + lb0 * wb0;
      l1 = l1 * wa1 + lb1 * wb1;
      m0 = M0;
      m1 = M1;
    }
  }

  if (p.n_splits == 1) {
    if (half == 0) {
      const float i0 = l0 > 0.f ? 1.f / l0 : 0.f, i1 = l1 > 0.f ? 1.f / l1 : 0.f;
      f16* out0 = p.out + ((size_t)(b * DFL_BLOCK + g) * hq + j) * D;
      f16* out1 = p.out + ((size_t)(b * DFL_BLOCK + g + 8) * hq + j) * D;
#pragma unroll
      for (int nd = 0; nd < D / 8; ++nd) {
        const int d = nd * 8 + 2 * c4;
        *reinterpret_cast<uint32_t*>(out0 + d) = pack_f16x2(o[nd][0] * i0, o[nd][1] * i0);
        *reinterpret_cast<uint32_t*>(out1 + d) = pack_f16x2(o[nd][2] * i1, o[nd][3] * i1);
      }
    }
    if (threadIdx.x == 0) atrace(p, 5);
    return;
  }

  // Splits of one (request, KV head) form a thread-block cluster: each CTA
  // leaves its partial in its own shared memory, the cluster barrier
  // publishes them, and CTA r merges rows r*rows/n .. of the output from all
  // partials over distributed shared memory, in split order -- every value a
  // thread needs (each split's max, sum and O piece) loaded at once.
  if (half == 0) {
#pragma unroll
    for (int nd = 0; nd < D / 8; ++nd) {
      const int d = nd * 8 + 2 * c4;
      *reinterpret_cast<float2*>(part + r0 * PS + d) = make_float2(o[nd][0], o[nd][1]);
      *reinterpret_cast<float2*>(part + r1 * PS + d) = make_float2(o[nd][2], o[nd][3]);
    }
    if (c4 == 0) {
      part[rows * PS + r0] = m0;
      part[rows * PS + r1] = m1;
      part[rows * PS + rows + r0] = l0;
      part[rows * PS + rows + r1] = l1;
    }
  }
  if (threadIdx.x == 0) atrace(p, 4);
  if (p.merge_global) {  // the partial goes to global memory; k_attn_merge combines the splits
    __syncthreads();
    copy_partial(p, part, rows * PS + 2 * rows, (b * hkv + kvh) * p.n_splits + split, D);
    if (threadIdx.x == 0) atrace(p, 5);
    return;
  }
  cluster_sync_all();

  const int n = p.n_splits;
  const int rank = (int)cluster_ctarank();
  const int rpc = (rows + n - 1) / n;  // rows merged by this CTA
  const int rb = rank * rpc, re = min(rows, rb + rpc);
  const uint32_t part_local = smem_u32(part);
  for (int e = threadIdx.x; e < (re - rb) * (D / 4); e += blockDim.x) {
    const int r = rb + e / (D / 4), d = (e % (D / 4)) * 4;
    float mv[ATTN_MAX_SPLITS], lv[ATTN_MAX_SPLITS];
    float4 v[ATTN_MAX_SPLITS];
#pragma unroll
    for (int sp = 0; sp < ATTN_MAX_SPLITS; ++sp) {
      mv[sp] = -INFINITY;
      lv[sp] = 0.f;
      v[sp] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (sp < n) {
        const uint32_t a = dsmem_addr(part_local, (uint32_t)sp);
        mv[sp] = ld_dsmem(a + 4u * (uint32_t)(rows * PS + r));
        lv[sp] = ld_dsmem(a + 4u * (uint32_t)(rows * PS + rows + r));
        v[sp] = ld_dsmem4(a + 4u * (uint32_t)(r * PS + d));
      }
    }
    float M = -INFINITY;
#pragma unroll
    for (int sp = 0; sp < ATTN_MAX_SPLITS; ++sp)
      if (lv[sp] > 0.f) M = fmaxf(M, mv[sp]);
    float L = 0.f;
#pragma unroll
    for (int sp = 0; sp < ATTN_MAX_SPLITS; ++sp) {
      const float w = lv[sp] > 0.f ? exp2f(mv[sp] - M) : 0.f;
      mv[sp] = w;
      L += w * lv[sp];
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int sp = 0; sp < ATTN_MAX_SPLITS; ++sp) {
      if (sp < n) {
        const float w = mv[sp] * inv;
        acc.x += w * v[sp].x;
        acc.y += w * v[sp].y;
        acc.z += w * v[sp].z;
        acc.w += w * v[sp].w;
      }
    }
    const int wq = r / 16, t = r % 16;
    f16* dst = p.out + ((size_t)(b * DFL_BLOCK + t) * hq + head0 + wq) * D + d;
    *reinterpret_cast<uint32_t*>(dst) = pack_f16x2(acc.x, acc.y);
    *reinterpret_cast<uint32_t*>(dst + 2) = pack_f16x2(acc.z, acc.w);
  }
  // keep this CTA's partial alive until every CTA of the cluster has read it
  cluster_sync_all();
  if (threadIdx.x == 0) atrace(p, 5);
}

// ---------------------------------------------------------------------------
// Block attention on the 5th-generation tensor cores.  Same grid, cluster,
// page split and merge as k_attn; per 64-key page:
//   S = Q K^T   tcgen05.mma M=128 (the G*16 query rows, zero-padded) x N=64 keys x K=D,
//   softmax     one query row per thread, read from TMEM, P written to shared
//               memory in the 128-byte-swizzle K-major layout,
//   O += P V    tcgen05.mma M=128 x N=D x K=64 keys, accumulated in TMEM.
// P is taken against a reference maximum that moves only when a page's row
// maximum exceeds it by more than 2^8 (then the row's O in TMEM is rescaled
// once), so P stays within f16 and O is read from TMEM only at the end; the
// result is the same softmax up to rounding.
// The K page is already the K-major B operand of the first MMA and the V^T
// page the K-major B operand of the second (pre-swizzled in HBM).  S is
// double-buffered, and the next page's Q K^T is issued before this page's
// P V, so the MMAs overlap the softmax.  A stage is refilled only once the
// P V of its page is done, so a CTA streams (stages) pages per (HBM round
// trip + page latency); measured per page on a 32K context: ~1.7 us from a
// load's issue to its landing, ~1.6 us from landing to the end of its P V.
// Q therefore lives in tensor memory (the S MMA's A operand) and P has a
// single buffer -- a page's P is written once the previous page's P V is
// done, by then long since, as P V is issued the moment P lands -- leaving
// shared memory to six 32 KB page stages.
// Warps: 0 page loads (one thread), 1 TMEM allocation and MMA issue (one
// thread), 2-9 softmax: two threads per query row (TMEM lane), each taking 32
// of a page's 64 keys and half of the output columns; the pair trades its
// half-row maxima through shared memory once per page.
template <int D>
struct TcCfg {
  static constexpr int STAGES = 6;                  // pages in flight
  static constexpr int BLK = 64 * D * 2;            // one K (or V^T) page block
  static constexpr int STAGE = 2 * BLK;
  static constexpr int PB = 128 * 64 * 2;           // P: 128 rows x 64 keys, one 16 KB panel
  static constexpr int OFF_P = STAGES * STAGE;     // one P buffer (Q lives in tensor memory)
  static constexpr int OFF_BAR = OFF_P + PB;
  static constexpr int MAX_PIDS = 512;
  static constexpr int OFF_PIDS = OFF_BAR + 256;
  static constexpr int OFF_X = OFF_PIDS + MAX_PIDS * 4;  // half-row exchange: [2 parities][2 halves][128] u64
  static constexpr int SMEM = 1024 + OFF_X + 2 * 2 * 128 * 8;  // + 1024 for aligning the base
  static constexpr int S_COL = 0;                   // S buffers: columns [0, 128)
  static constexpr int O_COL = 128;                 // O accumulator: columns [128, 128 + D)
  static constexpr int Q_COL = 256;                 // Q (tensor-memory A operand): columns [256, 256 + D/2)
  // columns allocated: a power of two covering the buffers, so two CTAs that
  // might share an SM never wait on each other's columns
  static constexpr uint32_t TMEM_COLS = 512;
};

// TMEM address of lane quarter q4 (lanes 32*q4 ..) at column 0.
DFL_DEV uint32_t lane_base_q(uint32_t tmem, int q4) { return tmem + ((uint32_t)(q4 * 32) << 16); }

template <int D, int G>
__global__ void __launch_bounds__(320, 1) k_attn_tc(const AttnParams p) {
  using C = TcCfg<D>;
  extern __shared__ __align__(128) uint8_t sm_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::OFF_BAR);
  uint64_t* full = bars;                    // [STAGES] page landed
  uint64_t* empty = full + C::STAGES;       // [STAGES] page's MMAs done
  uint64_t* s_full = empty + C::STAGES;     // [2] S in TMEM
  uint64_t* s_empty = s_full + 2;           // [2] S read by the softmax warps
  uint64_t* p_full = s_empty + 2;           // P of page i (phase i & 1) in shared memory
  uint64_t* o_full = p_full + 2;            // [2] P V of page i (barrier i & 1) complete
  uint64_t* q_full = o_full + 2;            // Q in tensor memory
  uint64_t* mdone = q_full + 1;             // every issued MMA complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mdone + 1);
  int* pids = reinterpret_cast<int*>(sm + C::OFF_PIDS);
  // xch[tag & 1][half][row] = (tag << 32) | float bits: the half-row value a
  // softmax thread publishes for its partner (tag = page index; n for the
  // final sum).  A thread cannot get two tags ahead of its partner (each
  // trade waits for the partner's same tag), so two parity slots suffice.
  volatile unsigned long long* xch = reinterpret_cast<volatile unsigned long long*>(sm + C::OFF_X);

  const int split = blockIdx.x, kvh = blockIdx.y, b = p.order ? p.order[blockIdx.z] : (int)blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rows = G * 16;
  for (int i = threadIdx.x; i < 512; i += blockDim.x) xch[i] = 0xFFFFFFFF00000000ull;  // no tag yet
  const int hq = p.hq, hkv = p.hkv;
  const uint32_t idesc_s = idesc_f16_f32(128, 64, 0);
  const uint32_t idesc_o = idesc_f16_f32(128, D, 0);

  if (threadIdx.x == 0) {
    atrace(p, 0);
    for (int i = 0; i < C::STAGES; ++i) {
      mbar_init(full + i, 1);
      mbar_init(empty + i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(s_full + i, 1);
      mbar_init(s_empty + i, 256);
      mbar_init(p_full + i, 256);
      mbar_init(o_full + i, 1);
    }
    mbar_init(q_full, 256);
    mbar_init(mdone, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_launch_dependents();
  if (!p.early) pdl_wait();

  const int slot = p.slots[b];
  const int nv = p.n_valid ? min(max(p.n_valid[b], 1), DFL_BLOCK) : p.block;  // live block rows
  const int nkeys = p.ctx_len[slot] + nv;             // context + live block rows
  const int ctx_pages = (nkeys - nv) >> 6;            // pages holding no block row
  const int npages = (nkeys + 63) >> 6;
  const int pb = (int)((long long)split * npages / p.n_splits);  // balanced page ranges
  const int pe = (int)((long long)(split + 1) * npages / p.n_splits);
  const int n = pe - pb;
  const int* pt = p.kv.page_table + (size_t)slot * p.kv.max_pages_per_slot;
  for (int i = threadIdx.x; i < n && i < C::MAX_PIDS; i += blockDim.x)
    pids[i] = pb + i < p.kv.max_pages_per_slot ? pt[pb + i] : -1;
  __syncthreads();
  if (threadIdx.x == 0) atrace(p, 1);
  bool aborted = false;

  // running state of this thread's half of a query row (softmax warps)
  constexpr int DH = D / 2;  // output columns per thread
  float o[DH];                           // set from TMEM after the last page
  float m_run = -INFINITY, l_run = 0.f;  // l_run: this half's keys only
  const int q4 = warp & 3;
  const int r = q4 * 32 + lane;        // TMEM lane = query row (softmax warps)
  const int kh = warp >= 6 ? 1 : 0;    // key / output-column half

  if (warp == 0) {
    // ------------------------------------------------ page loads
    if (lane == 0) {
      const f16* kbase = p.kv.k_pool + (size_t)p.layer * p.kv.layer_stride;
      const f16* vbase = p.kv.v_pool + (size_t)p.layer * p.kv.layer_stride;
      auto page_of_idx = [&](int i) {
        const int page_idx = pb + i;
        int pg = i < C::MAX_PIDS ? pids[i] : (page_idx < p.kv.max_pages_per_slot ? pt[page_idx] : -1);
        return (pg < 0 || pg >= p.kv.max_pages) ? -1 : pg;
      };
      int i = 0;
      bool waited = !p.early;
      for (; i < n; ++i) {
        const int s = i % C::STAGES;
        if (i >= C::STAGES && !mbar_wait(empty + s, (uint32_t)((i / C::STAGES - 1) & 1), p.status, &aborted)) break;
        if (!waited && pb + i >= ctx_pages) {  // the block's pages: written by the QKV projection
          pdl_wait();
          waited = true;
        }
        int pg = page_of_idx(i);
        if (pg < 0) {
          dev_error(p.status, DFLASH_DEV_PAGE);
          pg = 0;
        }
        const size_t off = ((size_t)pg * hkv + kvh) * (64 * D);
        uint8_t* dst = sm + s * C::STAGE;
        mbar_arrive_expect_tx(full + s, C::STAGE);
        bulk_load(dst, kbase + off, C::BLK, full + s);
        bulk_load(dst + C::BLK, vbase + off, C::BLK, full + s);
      }
      // every issued copy lands before the CTA may exit
      for (int j = (i > C::STAGES ? i - C::STAGES : 0); j < i; ++j) {
        bool drain_abort = false;
        mbar_wait(full + (j % C::STAGES), (uint32_t)((j / C::STAGES) & 1), p.status, &drain_abort);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issue
    // The whole warp runs the loop, converged (waits made warp-uniform), and
    // one elected lane issues each MMA and commit.
    auto wait_all = [&](uint64_t* bar, uint32_t par) {
      const bool ok = __all_sync(0xffffffffu, mbar_wait(bar, par, p.status, &aborted));
      if (!ok) aborted = true;
      return ok;
    };
    if (wait_all(q_full, 0)) {
      tc_fence_after();
      auto issue_s = [&](int i) {
        const int s = i % C::STAGES, bb = i & 1;
        if (!wait_all(full + s, (uint32_t)((i / C::STAGES) & 1))) return false;
        if (i >= 2 && !wait_all(s_empty + bb, (uint32_t)((i / 2 - 1) & 1))) return false;
        tc_fence_after();
        const uint32_t k_addr = smem_u32(sm + s * C::STAGE);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t bd = sdesc_sw128(k_addr + (uint32_t)((kk >> 2) * 8192)) + (uint64_t)(2 * (kk & 3));
          tc_mma_f16_ts_elect(tmem + (uint32_t)(C::S_COL + 64 * bb), tmem + (uint32_t)(C::Q_COL + 8 * kk), bd, idesc_s,
                              kk > 0 ? 1u : 0u);
        }
        tc_commit_elect(s_full + bb);
        return true;
      };
      bool ok = n == 0 || issue_s(0);
      for (int i = 0; i < n && ok; ++i) {
        if (i + 1 < n && !issue_s(i + 1)) break;
        const int s = i % C::STAGES, bb = i & 1;
        if (!wait_all(p_full, (uint32_t)(i & 1))) break;
        tc_fence_after();
        const uint32_t p_addr = smem_u32(sm + C::OFF_P);
        const uint32_t v_addr = smem_u32(sm + s * C::STAGE + C::BLK);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t ad = sdesc_sw128(p_addr) + (uint64_t)(2 * kk);
          const uint64_t bd = sdesc_sw128(v_addr) + (uint64_t)(2 * kk);
          tc_mma_f16_elect(tmem + (uint32_t)C::O_COL, ad, bd, idesc_o, (i > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit_elect(o_full + bb);
        tc_commit_elect(empty + s);
      }
      // every MMA this warp issued completes before the columns are freed
      tc_commit_elect(mdone);
      bool drain_abort = false;
      mbar_wait(mdone, 0, p.status, &drain_abort);
    }
  } else {
    // ------------------------------------------------ softmax (threads kh=0,1 of query row r)
    // trade a half-row value with the partner thread: publish ours under
    // `tag`, spin (bounded) until the partner's carries the same tag
    auto trade = [&](float mine, uint32_t tag, float* theirs) {
      const int slot0 = (int)(tag & 1u) * 256;
      xch[slot0 + kh * 128 + r] = ((unsigned long long)tag << 32) | __float_as_uint(mine);
      const uint64_t t0 = globaltimer();
      for (;;) {
        const unsigned long long v = xch[slot0 + (1 - kh) * 128 + r];
        if ((uint32_t)(v >> 32) == tag) {
          *theirs = __uint_as_float((uint32_t)v);
          return true;
        }
        if (globaltimer() - t0 > DFL_WAIT_NS) {
          dev_error(p.status, DFLASH_DEV_TIMEOUT);
          aborted = true;
          return false;
        }
      }
    };
    if (p.early) pdl_wait();  // the queries come from the QKV projection
    {  // this row's query (half of its chunks per thread), zero-padded to 128 rows
      const int h = r >> 4, t = r & 15;
      const f16* src = p.q + ((size_t)(b * DFL_BLOCK + t) * hq + kvh * G + h) * D;
      // TMEM lane r, columns Q_COL + kh*D/4 ...: two f16 per column
      uint4 v[D / 16];
#pragma unroll
      for (int cc = 0; cc < D / 16; ++cc)
        v[cc] = r < rows ? *reinterpret_cast<const uint4*>(src + (kh * (D / 16) + cc) * 8) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int j = 0; j < D / 64; ++j)
        tmem_st16(lane_base_q(tmem, q4) + (uint32_t)(C::Q_COL + kh * (D / 4) + 16 * j),
                  reinterpret_cast<const float*>(&v[4 * j]));
      tc_fence_before();
      mbar_arrive(q_full);
    }
    const uint32_t lane_base = tmem + ((uint32_t)(q4 * 32) << 16);
    // this row's keys: all, or (causal) the context and block rows up to the
    // row's own token (padding rows: up to the last live row)
    const int klim = p.causal ? nkeys - nv + min(r & 15, nv - 1) + 1 : nkeys;
    // P V of page i complete (o_full[i & 1]).  Waited once per page, before
    // P of the next page is written (one P buffer), so a barrier never runs
    // two phases ahead of its waiter.
    int o_seen = -1;  // pages whose P V this thread has seen complete
    auto wait_o = [&](int i) {
      if (i <= o_seen) return true;
      if (!mbar_wait(o_full + (i & 1), (uint32_t)((i / 2) & 1), p.status, &aborted)) return false;
      o_seen = i;
      return true;
    };
    bool ok = true;
    for (int i = 0; i < n && ok; ++i) {
      const int bb = i & 1;
      if (!mbar_wait(s_full + bb, (uint32_t)((i / 2) & 1), p.status, &aborted)) break;
      if (i == 0 && threadIdx.x == 64) atrace(p, 2);
      tc_fence_after();
      float sc[32];
      {
        uint32_t u[32];
#pragma unroll
        for (int j = 0; j < 2; ++j)
          tmem_ld16_nowait(lane_base + (uint32_t)(C::S_COL + 64 * bb + 32 * kh + 16 * j), u + 16 * j);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 32; ++k) sc[k] = __uint_as_float(u[k]);
      }
      tc_fence_before();
      mbar_arrive(s_empty + bb);
      const int valid = min(64, klim - (pb + i) * 64) - 32 * kh;  // this half's unmasked keys
      float mx = -INFINITY;
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        sc[k] = k < valid ? sc[k] * p.scale_log2 : -INFINITY;
        mx = fmaxf(mx, sc[k]);
      }
      float mx_other;
      if (!trade(mx, (uint32_t)i, &mx_other)) break;
      const float mx_all = fmaxf(mx, mx_other);
      const bool move = mx_all > m_run + 8.f;  // same decision in both threads of the row
      if (__any_sync(0xffffffffu, move)) {     // TMEM access is warp-wide
        const float m_new = move ? mx_all : m_run;
        if (i > 0) {  // O holds pages < i against m_run: rescale it once P V of page i-1 is done
          if (!wait_o(i - 1)) break;
          tc_fence_after();
          const float alpha = move ? exp2f(m_run - m_new) : 1.f;
#pragma unroll
          for (int j = 0; j < DH / 16; ++j) {
            float v[16];
            const uint32_t ta = lane_base + (uint32_t)(C::O_COL + kh * DH + 16 * j);
            tmem_ld16(ta, v);
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] *= alpha;
            tmem_st16(ta, v);
          }
          tc_fence_before();
          l_run *= alpha;
        }
        m_run = m_new;
      }
      const float ref = m_run == -INFINITY ? 0.f : m_run;  // a row with only masked keys so far adds 0
      float rs = 0.f;
      uint32_t pk[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const float a = exp2f(sc[2 * k] - ref), c = exp2f(sc[2 * k + 1] - ref);
        rs += a + c;
        pk[k] = pack_f16x2(a, c);
      }
      l_run += rs;
      if (i > 0 && !wait_o(i - 1)) break;  // the previous page's P V has read the P buffer
      {  // this half of P row r: 32 keys = 4 chunks of 16 bytes, swizzled like the K page rows
        uint8_t* prow = sm + C::OFF_P + r * 128;
#pragma unroll
        for (int c = 0; c < 4; ++c)
          *reinterpret_cast<uint4*>(prow + ((((4 * kh + c) ^ (r & 7))) << 4)) =
              make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      }
      fence_proxy_async_smem();
      mbar_arrive(p_full);
    }
    // the row's output half, once every P V is done
    if (ok && n > 0 && !aborted && wait_o(n - 1)) {
      tc_fence_after();
#pragma unroll
      for (int j = 0; j < DH / 16; ++j) tmem_ld16(lane_base + (uint32_t)(C::O_COL + kh * DH + 16 * j), o + 16 * j);
    } else {
#pragma unroll
      for (int d = 0; d < DH; ++d) o[d] = 0.f;
    }
    // the row's sum over both halves
    float l_other = 0.f;
    if (!aborted && trade(l_run, (uint32_t)n, &l_other)) l_run += l_other;
  }
  if (threadIdx.x == 0) atrace(p, 3);
  tc_fence_before();
  __syncthreads();  // every TMEM read and MMA done, every page landed
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }

  const int h = r >> 4, t = r & 15;
  const bool row_out = warp >= 2 && r < rows;
  if (p.n_splits == 1) {
    if (row_out) {
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      f16* dst = p.out + ((size_t)(b * DFL_BLOCK + t) * hq + kvh * G + h) * D + kh * DH;
#pragma unroll
      for (int c = 0; c < DH / 8; ++c)
        *reinterpret_cast<uint4*>(dst + c * 8) =
            make_uint4(pack_f16x2(o[8 * c] * inv, o[8 * c + 1] * inv), pack_f16x2(o[8 * c + 2] * inv, o[8 * c + 3] * inv),
                       pack_f16x2(o[8 * c + 4] * inv, o[8 * c + 5] * inv), pack_f16x2(o[8 * c + 6] * inv, o[8 * c + 7] * inv));
    }
    if (threadIdx.x == 0) atrace(p, 5);
    return;
  }

  // partial (unnormalised O, running max, running sum) for the cluster merge,
  // in the page-stage area (every page is consumed)
  constexpr int PS = D + 4;
  float* part = reinterpret_cast<float*>(sm);
  if (row_out) {
#pragma unroll
    for (int c = 0; c < DH / 4; ++c)
      *reinterpret_cast<float4*>(part + r * PS + kh * DH + 4 * c) =
          make_float4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
    if (kh == 0) {
      part[rows * PS + r] = m_run;
      part[rows * PS + rows + r] = l_run;
    }
  }
  if (threadIdx.x == 0) atrace(p, 4);
  if (p.merge_global) {  // the partial goes to global memory; k_attn_merge combines the splits
    __syncthreads();
    copy_partial(p, part, rows * PS + 2 * rows, (b * hkv + kvh) * p.n_splits + split, D);
    if (threadIdx.x == 0) atrace(p, 5);
    return;
  }
  cluster_sync_all();

  const int nsp = p.n_splits;
  const int rank = (int)cluster_ctarank();
  const int rpc = (rows + nsp - 1) / nsp;  // rows merged by this CTA
  const int rb = rank * rpc, re = min(rows, rb + rpc);
  const uint32_t part_local = smem_u32(part);
  for (int e = threadIdx.x; e < (re - rb) * (D / 4); e += blockDim.x) {
    const int rr = rb + e / (D / 4), d = (e % (D / 4)) * 4;
    float mv[ATTN_MAX_SPLITS], lv[ATTN_MAX_SPLITS];
    float4 v[ATTN_MAX_SPLITS];
#pragma unroll
    for (int sp = 0; sp < ATTN_MAX_SPLITS; ++sp) {
      mv[sp] = -INFINITY;
      lv[sp] = 0.f;
      v[sp] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (sp < nsp) {
        const uint32_t a = dsmem_addr(part_local, (uint32_t)sp);
        mv[sp] = ld_dsmem(a + 4u * (uint32_t)(rows * PS + rr));
        lv[sp] = ld_dsmem(a + 4u * (uint32_t)(rows * PS + rows + rr));
        v[sp] = ld_dsmem4(a + 4u * (uint32_t)(rr * PS + d));
      }
    }
    float M = -INFINITY;
#pragma unroll
    for (int sp = 0; sp < ATTN_MAX_SPLITS; ++sp)
      if (lv[sp] > 0.f) M = fmaxf(M, mv[sp]);
    float L = 0.f;
#pragma unroll
    for (int sp = 0; sp < ATTN_MAX_SPLITS; ++sp) {
      const float w = lv[sp] > 0.f ? exp2f(mv[sp] - M) : 0.f;
      mv[sp] = w;
      L += w * lv[sp];
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int sp = 0; sp < ATTN_MAX_SPLITS; ++sp) {
      if (sp < nsp) {
        const float w = mv[sp] * inv;
        acc.x += w * v[sp].x;
        acc.y += w * v[sp].y;
        acc.z += w * v[sp].z;
        acc.w += w * v[sp].w;
      }
    }
    const int wq = rr / 16, tt = rr % 16;
    f16* dst = p.out + ((size_t)(b * DFL_BLOCK + tt) * hq + kvh * G + wq) * D + d;
    *reinterpret_cast<uint32_t*>(dst) = pack_f16x2(acc.x, acc.y);
    *reinterpret_cast<uint32_t*>(dst + 2) = pack_f16x2(acc.z, acc.w);
  }
  // keep this CTA's partial alive until every CTA of the cluster has read it
  cluster_sync_all();
  if (threadIdx.x == 0) atrace(p, 5);
}

// key split per head: 2 warps per query head up to 4 heads per KV head
template <int G>
constexpr int attn_ks() {
  return G <= 4 ? 2 : 1;
}

// The kernel instance, block size and shared memory of one page loop for (D, G).
template <int D, int G, bool TC>
struct AttnKernel;
template <int D, int G>
struct AttnKernel<D, G, true> {
  static constexpr auto fn = k_attn_tc<D, G>;
  static constexpr int threads = 320;
  static constexpr int smem = TcCfg<D>::SMEM;
};
template <int D, int G>
struct AttnKernel<D, G, false> {
  static constexpr auto fn = k_attn<D, G, attn_ks<G>()>;
  static constexpr int threads = G * attn_ks<G>() * 32;
  static constexpr int smem = AttnCfg<D>::SMEM;
};

template <int D, int G, bool TC>
cudaError_t launch_t(const AttnParams& p, int batch, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.n_splits, (unsigned)p.hkv, (unsigned)batch);
  cfg.blockDim = dim3(AttnKernel<D, G, TC>::threads);
  cfg.dynamicSmemBytes = AttnKernel<D, G, TC>::smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (!p.merge_global) {
    attr[na].id = cudaLaunchAttributeClusterDimension;  // the splits of one KV head
    attr[na].val.clusterDim.x = (unsigned)p.n_splits;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = (unsigned)na;
  cudaError_t e = cudaLaunchKernelEx(&cfg, AttnKernel<D, G, TC>::fn, p);
  if (e || !p.merge_global || p.n_splits == 1) return e;
  cudaLaunchConfig_t mc = {};
  mc.gridDim = dim3((unsigned)(batch * p.hkv), (unsigned)G);  // 16 rows per CTA
  mc.blockDim = dim3(16 * MERGE_TPR);
  mc.stream = s;
  mc.attrs = attr + na - (pdl ? 1 : 0);
  mc.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&mc, k_attn_merge<D>, p);
}

template <int D, bool TC>
cudaError_t launch_d(const AttnParams& p, int batch, cudaStream_t s, bool pdl) {
  switch (p.hq / p.hkv) {
    case 1: return launch_t<D, 1, TC>(p, batch, s, pdl);
    case 2: return launch_t<D, 2, TC>(p, batch, s, pdl);
    case 4: return launch_t<D, 4, TC>(p, batch, s, pdl);
    case 8: return launch_t<D, 8, TC>(p, batch, s, pdl);
  }
  return cudaErrorInvalidValue;
}

template <int D, int G, bool TC>
cudaError_t attr_t() {
  auto k = AttnKernel<D, G, TC>::fn;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, AttnKernel<D, G, TC>::smem);
  if (e) return e;
  return cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
}

template <int D, bool TC>
cudaError_t attr_d() {
  cudaError_t e;
  if ((e = attr_t<D, 1, TC>())) return e;
  if ((e = attr_t<D, 2, TC>())) return e;
  if ((e = attr_t<D, 4, TC>())) return e;
  return attr_t<D, 8, TC>();
}

// Clusters of `splits` CTAs of the attention kernel for this shape that the
// GPU can hold at once (0 when it cannot launch them at all).
template <int D, int G, bool TC>
int max_clusters_t(int splits, int hkv) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)splits, (unsigned)hkv, 1);
  cfg.blockDim = dim3(AttnKernel<D, G, TC>::threads);
  cfg.dynamicSmemBytes = AttnKernel<D, G, TC>::smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)splits;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, AttnKernel<D, G, TC>::fn, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

template <int D, bool TC>
int max_clusters_d(int splits, int G, int hkv) {
  switch (G) {
    case 1: return max_clusters_t<D, 1, TC>(splits, hkv);
    case 2: return max_clusters_t<D, 2, TC>(splits, hkv);
    case 4: return max_clusters_t<D, 4, TC>(splits, hkv);
    case 8: return max_clusters_t<D, 8, TC>(splits, hkv);
  }
  return 0;
}

}  // namespace

int attn_max_active_clusters(int D, int hq, int hkv, int splits, bool tc) {
  if (splits < 1 || splits > ATTN_MAX_SPLITS) return 0;
  const int G = hq / hkv;
  if (D == 64) return tc ? max_clusters_d<64, true>(splits, G, hkv) : max_clusters_d<64, false>(splits, G, hkv);
  return tc ? max_clusters_d<128, true>(splits, G, hkv) : max_clusters_d<128, false>(splits, G, hkv);
}

cudaError_t attn_init_attributes() {
  cudaError_t e;
  if ((e = attr_d<64, false>())) return e;
  if ((e = attr_d<64, true>())) return e;
  if ((e = attr_d<128, false>())) return e;
  return attr_d<128, true>();
}

cudaError_t attn_launch(const AttnParams& p, int batch, cudaStream_t s, bool pdl, bool tc) {
  if (p.D == 64) return tc ? launch_d<64, true>(p, batch, s, pdl) : launch_d<64, false>(p, batch, s, pdl);
  if (p.D == 128) return tc ? launch_d<128, true>(p, batch, s, pdl) : launch_d<128, false>(p, batch, s, pdl);
  return cudaErrorInvalidValue;
}
