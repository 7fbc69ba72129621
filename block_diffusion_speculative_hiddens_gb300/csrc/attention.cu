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
// length known, 2 first page landed, 3 pages done, 4 partial published, 5 exit.
DFL_DEV void atrace(const AttnParams& p, int ev) {
  if (p.trace) {
    const size_t cta = ((size_t)blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
    p.trace[cta * 8 + ev] = globaltimer();
  }
}

// KS warps per query head split every page's 64 keys between them (KS = 2
// for G <= 4), each with its own online softmax, merged in shared memory at
// the end: twice the warps in flight and half the dependent MMA chain per
// page for the common GQA group sizes.
template <int D, int G, int KS>
__global__ void __launch_bounds__(G * KS * 32) k_attn(const AttnParams p) {
  using C = AttnCfg<D>;
  constexpr int KPW = 64 / KS;   // keys of a page per warp
  constexpr int NKG = KPW / 16;  // 16-key groups per warp
  constexpr int PS = D + 4;      // padded row stride (floats) of a partial
  extern __shared__ __align__(128) uint8_t sm[];
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + C::STAGES * C::STAGE_BYTES);
  int* pids = reinterpret_cast<int*>(sm + C::STAGES * C::STAGE_BYTES + 128);

  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
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
  pdl_wait();

  const int slot = p.slots[b];
  const int nkeys = p.ctx_len[slot] + DFL_BLOCK;
  const int npages = (nkeys + 63) >> 6;
  const int pb = (int)((long long)split * npages / p.n_splits);  // balanced page ranges
  const int pe = (int)((long long)(split + 1) * npages / p.n_splits);
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
  if (threadIdx.x == 0)
    for (int i = 0; i < C::STAGES && pb + i < pe; ++i, ++issued) issue(i, pb + i);

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
      const int valid = min(64, nkeys - pi * 64);
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
          if (key >= valid) v = -INFINITY;
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

// key split per head: 2 warps per query head up to 4 heads per KV head
template <int G>
constexpr int attn_ks() {
  return G <= 4 ? 2 : 1;
}

template <int D, int G>
cudaError_t launch_t(const AttnParams& p, int batch, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.n_splits, (unsigned)p.hkv, (unsigned)batch);
  cfg.blockDim = dim3(G * attn_ks<G>() * 32);
  cfg.dynamicSmemBytes = AttnCfg<D>::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;  // the splits of one KV head
  attr[0].val.clusterDim.x = (unsigned)p.n_splits;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, k_attn<D, G, attn_ks<G>()>, p);
}

template <int D>
cudaError_t launch_d(const AttnParams& p, int batch, cudaStream_t s, bool pdl) {
  switch (p.hq / p.hkv) {
    case 1: return launch_t<D, 1>(p, batch, s, pdl);
    case 2: return launch_t<D, 2>(p, batch, s, pdl);
    case 4: return launch_t<D, 4>(p, batch, s, pdl);
    case 8: return launch_t<D, 8>(p, batch, s, pdl);
  }
  return cudaErrorInvalidValue;
}

template <int D, int G>
cudaError_t attr_t() {
  auto k = k_attn<D, G, attn_ks<G>()>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, AttnCfg<D>::SMEM);
  if (e) return e;
  return cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
}

template <int D>
cudaError_t attr_d() {
  cudaError_t e;
  if ((e = attr_t<D, 1>())) return e;
  if ((e = attr_t<D, 2>())) return e;
  if ((e = attr_t<D, 4>())) return e;
  return attr_t<D, 8>();
}

// Clusters of `splits` CTAs of the attention kernel for this shape that the
// GPU can hold at once (0 when it cannot launch them at all).
template <int D, int G>
int max_clusters_t(int splits, int hkv) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)splits, (unsigned)hkv, 1);
  cfg.blockDim = dim3(G * attn_ks<G>() * 32);
  cfg.dynamicSmemBytes = AttnCfg<D>::SMEM;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)splits;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, k_attn<D, G, attn_ks<G>()>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

template <int D>
int max_clusters_d(int splits, int G, int hkv) {
  switch (G) {
    case 1: return max_clusters_t<D, 1>(splits, hkv);
    case 2: return max_clusters_t<D, 2>(splits, hkv);
    case 4: return max_clusters_t<D, 4>(splits, hkv);
    case 8: return max_clusters_t<D, 8>(splits, hkv);
  }
  return 0;
}

}  // namespace

size_t attn_smem_bytes(int D) { return D == 64 ? AttnCfg<64>::SMEM : AttnCfg<128>::SMEM; }

int attn_max_active_clusters(int D, int hq, int hkv, int splits) {
  if (splits < 1 || splits > ATTN_MAX_SPLITS) return 0;
  return D == 64 ? max_clusters_d<64>(splits, hq / hkv, hkv) : max_clusters_d<128>(splits, hq / hkv, hkv);
}

cudaError_t attn_init_attributes() {
  cudaError_t e = attr_d<64>();
  if (e) return e;
  return attr_d<128>();
}

cudaError_t attn_launch(const AttnParams& p, int batch, cudaStream_t s, bool pdl) {
  if (p.D == 64) return launch_d<64>(p, batch, s, pdl);
  if (p.D == 128) return launch_d<128>(p, batch, s, pdl);
  return cudaErrorInvalidValue;
}
