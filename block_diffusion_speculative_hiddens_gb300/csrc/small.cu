// Small kernels of the round: block embedding, page allocation, acceptance,
// slot reset, RoPE table, cache read-back and the benchmark's stand-in verify.
#include <algorithm>

#include <cuda_fp8.h>

#include "common.cuh"
#include "internal.h"

namespace {

cudaLaunchConfig_t cfg_of(dim3 grid, dim3 block, cudaStream_t s, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t c = {};
  c.gridDim = grid;
  c.blockDim = block;
  c.stream = s;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  c.attrs = attr;
  c.numAttrs = 1;
  return c;
}

// Weight preparation: row-major bf16 [N, K] -> packed blocks of 128 rows x 64
// columns ([tile][k-block]), each in the 128-byte-swizzle image, converted to
// f16 (exact for every bf16 value in the f16 normal range) or kept bf16.
// swiglu_I > 0 packs a [2I, K] gate/up matrix so that tile t holds gate rows
// t*64..t*64+63 then up rows I+t*64..I+t*64+63.  Rows past N are zero.  A
// weight beyond the f16 range (|w| > 65504) is saturated and sets
// DFLASH_DEV_RANGE, which dflash_create turns into DFLASH_ERR_RANGE.
__global__ void k_pack_weight(const bf16* __restrict__ src, uint16_t* __restrict__ dst, int N, int K, int n_tiles,
                              int swiglu_I, int conv, uint32_t* status) {
  const int KB = K / 64;
  const long long total = (long long)n_tiles * KB * 128 * 8;  // 16-byte chunks
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const int c = (int)(idx & 7);
    const int r = (int)((idx >> 3) & 127);
    const long long blk = idx >> 10;
    const int tile = (int)(blk / KB), kb = (int)(blk % KB);
    const int row = swiglu_I > 0 ? (r < 64 ? tile * 64 + r : swiglu_I + tile * 64 + (r - 64)) : tile * 128 + r;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (row < N) v = *reinterpret_cast<const uint4*>(src + (size_t)row * K + kb * 64 + c * 8);
    if (conv) {
      const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&v);
      uint4 o;
      __half2* h2 = reinterpret_cast<__half2*>(&o);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(b2[i]);
        h2[i] = __halves2half2(to_f16(f.x, status), to_f16(f.y, status));
      }
      v = o;
    }
    *reinterpret_cast<uint4*>(dst + blk * DFL_WBLK_ELEMS + r * 64 + ((c ^ (r & 7)) << 3)) = v;
  }
}

// FP8 packing, pass 1: one warp per packed row -- the row's scale
// max|w| / 448 (1 for an all-zero or padding row).
__global__ void k_fp8_scale(const bf16* __restrict__ src, float* __restrict__ scale, int N, int K, int n_rows,
                            int swiglu_I) {
  const int pr = (int)((blockIdx.x * (unsigned)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (pr >= n_rows) return;
  const int tile = pr >> 7, r = pr & 127;
  const int row = swiglu_I > 0 ? (r < 64 ? tile * 64 + r : swiglu_I + tile * 64 + (r - 64)) : pr;
  float m = 0.f;
  if (row < N)
    for (int k = lane; k < K; k += 32) m = fmaxf(m, fabsf(__bfloat162float(src[(size_t)row * K + k])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) scale[pr] = m > 0.f ? __fdiv_rn(m, 448.f) : 1.f;
}

// FP8 packing, pass 2: 16 weights per thread, w / scale (correctly rounded)
// to E4M3 (nearest even, saturating), blocks of 128 rows x 64 bytes.
__global__ void k_pack_fp8(const bf16* __restrict__ src, const float* __restrict__ scale, uint8_t* __restrict__ dst,
                           int N, int K, int n_tiles, int swiglu_I) {
  const int KB = K / 64;
  const long long total = (long long)n_tiles * KB * 128 * 4;  // 16-value chunks
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const int c = (int)(idx & 3);
    const int r = (int)((idx >> 2) & 127);
    const long long blk = idx >> 9;
    const int tile = (int)(blk / KB), kb = (int)(blk % KB);
    const int row = swiglu_I > 0 ? (r < 64 ? tile * 64 + r : swiglu_I + tile * 64 + (r - 64)) : tile * 128 + r;
    uint8_t q[16];
    const float sc = scale[tile * 128 + r];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float w = row < N ? __bfloat162float(src[(size_t)row * K + kb * 64 + c * 16 + i]) : 0.f;
      q[i] = (uint8_t)__nv_cvt_float_to_fp8(__fdiv_rn(w, sc), __NV_SATFINITE, __NV_E4M3);
    }
    *reinterpret_cast<uint4*>(dst + blk * DFL_WBLK8_BYTES + r * 64 + c * 16) = *reinterpret_cast<const uint4*>(q);
  }
}

__global__ void k_gain_f32(const bf16* __restrict__ src, float* __restrict__ dst, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) dst[i] = __bfloat162float(src[i]);
}

// a3: block = [last_tok, mask x 15]; h = E[block] (fp32 residual stream, read
// from the packed f16 table), hg = f16(h * g_in0) and per-128-feature sums of
// squares of h, the form the first layer's QKV GEMM consumes.  Also clears
// the argmax keys.
__global__ void k_embed(const int* __restrict__ slots, const int* __restrict__ last_tok, int mask_id, int vocab,
                        const void* __restrict__ Ev, const float* __restrict__ escale, const float* __restrict__ gain,
                        int H, int M, float* h, f16* hg, float* ss, unsigned long long* keys, const BlockCtx bc,
                        uint32_t* status) {
  pdl_launch_dependents();
  pdl_wait();
  const int t = blockIdx.x;
  const int b = t / DFL_BLOCK, i = t % DFL_BLOCK;
  int nv = bc.n_valid ? bc.n_valid[b] : bc.block;  // live rows of this request
  if (nv < 1 || nv > DFL_BLOCK) {
    if (threadIdx.x == 0 && i == 0) dev_error(status, DFLASH_DEV_ARG);
    nv = nv < 1 ? 1 : DFL_BLOCK;
  }
  int tok = bc.tokens ? (i < nv ? bc.tokens[t] : mask_id) : (i == 0 ? last_tok[b] : mask_id);
  if (tok < 0 || tok >= vocab) {
    if (threadIdx.x == 0) dev_error(status, DFLASH_DEV_ARG);
    tok = mask_id;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const int KB = H / 64;
  const int r = tok & 127;
  // the tied table: packed f16 blocks, or FP8 blocks (row-major) with a scale per vocabulary row
  const f16* tile = static_cast<const f16*>(Ev) + (size_t)(tok >> 7) * KB * DFL_WBLK_ELEMS;
  const uint8_t* tile8 = static_cast<const uint8_t*>(Ev) + (size_t)(tok >> 7) * KB * DFL_WBLK8_BYTES;
  const float es = escale ? escale[tok] : 1.f;
  for (int part = warp; part < H / 128; part += nw) {
    float sq = 0.f;
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      const int n = part * 128 + lane + 32 * jj;
      const float v = escale ? __half2float(__ushort_as_half((unsigned short)(e4m3x2_to_f16x2(
                                   tile8[(size_t)(n >> 6) * DFL_WBLK8_BYTES + r * 64 + (n & 63)]) & 0xFFFFu))) * es
                             : __half2float(tile[(size_t)(n >> 6) * DFL_WBLK_ELEMS + wpack_off(r, n & 63)]);
      h[(size_t)t * H + n] = v;
      hg[(size_t)t * H + n] = to_f16(v * gain[n], status);
      sq += v * v;
    }
    sq = warp_sum(sq);
    if (lane == 0) ss[(size_t)part * M + t] = sq;
  }
  if (threadIdx.x == 0) keys[t] = 0ull;
  if (bc.order && t == 0) {
    // the requests by descending context length (ties: request order), for
    // the attention grid: request j's rank is the count of requests that
    // come before it
    const int batch = M / DFL_BLOCK;
    for (int j = threadIdx.x; j < batch; j += blockDim.x) {
      const int sj = slots[j];
      const int lj = (sj >= 0 && sj < bc.max_slots) ? bc.ctx_len[sj] : 0;
      int rank = 0;
      for (int k = 0; k < batch; ++k) {
        const int sk = slots[k];
        const int lk = (sk >= 0 && sk < bc.max_slots) ? bc.ctx_len[sk] : 0;
        rank += (lk > lj || (lk == lj && k < j)) ? 1 : 0;
      }
      bc.order[rank] = j;
    }
  }
  // this token's position (block rows follow the slot's context), page and
  // RoPE row, for every layer's QKV epilogue
  // rows block..15 of a request pad a smaller block: page -2 (computed like
  // any row, at a position clamped into the table, but never written to the
  // cache, so they never become keys).  A request with an out-of-range slot
  // is reported, read from slot 0 and written nowhere (all rows padding).
  const int slot_in = slots[b];
  const bool bad_slot = slot_in < 0 || slot_in >= bc.max_slots;
  const int slot = bad_slot ? 0 : slot_in;
  if (i == 0 && threadIdx.x == 0) {
    bc.slots_ok[b] = slot;
    if (bad_slot) dev_error(status, DFLASH_DEV_ARG);
  }
  const bool pad = i >= nv || bad_slot;
  const int pos = pad ? min(bc.ctx_len[slot] + i, bc.max_pos - 1) : bc.ctx_len[slot] + i;
  const bool in_range = pos < bc.max_pos;
  if (threadIdx.x == 0) {
    int pg = -1;
    if (pad) {
      pg = -2;
    } else if (!in_range) {
      dev_error(status, DFLASH_DEV_CAPACITY);
    } else if ((pos >> 6) < bc.max_pages_per_slot) {
      pg = bc.page_table[(size_t)slot * bc.max_pages_per_slot + (pos >> 6)];
      if (pg < 0 || pg >= bc.max_pages) pg = -1;
    }
    bc.bctx[t] = make_int2(pos, pg);
  }
  for (int k = threadIdx.x; k < bc.D / 2; k += blockDim.x)
    bc.brope[(size_t)t * (bc.D / 2) + k] = in_range ? bc.rope[(size_t)pos * (bc.D / 2) + k] : make_float2(1.f, 0.f);
}

// Page allocation for dflash_fuse_inject (one thread, requests in order, so
// the page assignment is deterministic).  Grows each slot's page table to
// cover ctx_len + n_new + block positions, records the first new position
// (pos0, per request) and the effective row count, and advances ctx_len.
// With row_off non-null it also gives each request's first row among the
// appended rows of all requests (row_off[b]) and their total (*n_live), for
// an injection over the appended rows alone.
__global__ void k_page_alloc(const int* slots, int batch, int S, const int* n_new, int rows_per_req, int* ctx_len,
                             int* pos0, int* n_pages, int* page_table, int mpps, int* free_stack, int* free_top,
                             int* n_eff, int* slots_ok, int max_slots, uint32_t* status, int* row_off,
                             int* n_live) {
  pdl_launch_dependents();
  pdl_wait();
  if (threadIdx.x != 0) return;
  int top = *free_top;
  int live = 0;
  for (int b = 0; b < batch; ++b) {
    const int slot = slots[b];
    if (slot < 0 || slot >= max_slots) {
      dev_error(status, DFLASH_DEV_ARG);
      n_eff[b] = 0;
      pos0[b] = 0;
      slots_ok[b] = 0;  // in bounds for the later kernels; no row of it is live
      if (row_off) row_off[b] = live;
      continue;
    }
    slots_ok[b] = slot;
    int n = n_new ? n_new[b] : 0;  // null: only pages for the next block
    if (n < 0 || n > rows_per_req) {
      dev_error(status, DFLASH_DEV_ARG);
      n = 0;
    }
    const int L = ctx_len[slot];
    int need = (L + n + S + DFL_PAGE - 1) / DFL_PAGE;
    if (need > mpps) {
      dev_error(status, DFLASH_DEV_CAPACITY);
      n = 0;
      need = min(mpps, (L + S + DFL_PAGE - 1) / DFL_PAGE);
    }
    int np = n_pages[slot];
    while (np < need) {
      if (top == 0) {
        dev_error(status, DFLASH_DEV_CAPACITY);
        break;
      }
      page_table[(size_t)slot * mpps + np] = free_stack[--top];
      ++np;
    }
    if (np * DFL_PAGE < L + n) n = 0;  // no room for the new rows
    n_pages[slot] = np;
    pos0[b] = L;
    ctx_len[slot] = L + n;
    n_eff[b] = n;
    if (row_off) row_off[b] = live;
    live += n;
  }
  *free_top = top;
  if (n_live) *n_live = live;
}

// One block per (row i, request b): the row is copied when it is appended.
__global__ void k_compact_rows(const bf16* __restrict__ feats, int rows_per_req, int F, const int* n_eff,
                               const int* row_off, bf16* __restrict__ dst, int* row_map) {
  pdl_launch_dependents();
  pdl_wait();
  const int i = blockIdx.x, b = blockIdx.y;
  if (i >= n_eff[b]) return;
  const int j = row_off[b] + i;
  const int src_row = b * rows_per_req + i;
  if (threadIdx.x == 0) row_map[j] = src_row;
  const uint4* s = reinterpret_cast<const uint4*>(feats + (size_t)src_row * F);
  uint4* d = reinterpret_cast<uint4*>(dst + (size_t)j * F);
  for (int k = threadIdx.x; k < F / 8; k += blockDim.x) d[k] = s[k];
}

// a7: one warp per request.  Lane i compares draft d_{i+1} with target t_i;
// the ballot's lowest zero bit is the first mismatch n, so the accepted
// prefix is the cumulative product of the matches; tau = n + 1, the bonus is
// t_n, and the confirmed length is ctx_len + tau.
__global__ void k_accept(const int* slots, int batch, int S, const int* draft, const int* target, int* accept_len,
                         int* bonus, int* ctx_out, const int* ctx_len, int max_slots, uint32_t* status) {
  pdl_launch_dependents();
  pdl_wait();
  const int b = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (b >= batch) return;
  const bool match = lane < S - 1 && draft[b * (S - 1) + lane] == target[b * S + lane];
  const unsigned m = __ballot_sync(0xffffffffu, match);
  const int n = __ffs(~m) - 1;  // bits S-1.. of m are 0, so n <= S-1
  if (lane == 0) {
    const int tau = n + 1;
    const int slot = slots[b];
    int L = 0;
    if (slot < 0 || slot >= max_slots)
      dev_error(status, DFLASH_DEV_ARG);
    else
      L = ctx_len[slot];
    accept_len[b] = tau;
    bonus[b] = target[b * S + n];
    ctx_out[b] = L + tau;
  }
}

__global__ void k_reset_slot(int slot, int* ctx_len, int* n_pages, int* page_table, int mpps, int* free_stack,
                             int* free_top) {
  pdl_launch_dependents();
  pdl_wait();
  if (threadIdx.x != 0) return;
  int top = *free_top;
  const int np = n_pages[slot];
  for (int i = np - 1; i >= 0; --i) {
    free_stack[top++] = page_table[(size_t)slot * mpps + i];
    page_table[(size_t)slot * mpps + i] = -1;
  }
  *free_top = top;
  n_pages[slot] = 0;
  ctx_len[slot] = 0;
}

__global__ void k_pool_init(int* free_stack, int* free_top, int max_pages) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < max_pages) free_stack[i] = max_pages - 1 - i;  // pops 0, 1, 2, ...
  if (i == 0) *free_top = max_pages;
}

// RoPE angles pos * theta^(-2i/D) evaluated in double precision, stored as
// float (cos, sin) pairs.
__global__ void k_rope_table(float2* tab, int max_pos, int D, double theta) {
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const int half = D / 2;
  if (idx >= (long long)max_pos * half) return;
  const int pos = (int)(idx / half), i = (int)(idx % half);
  const double inv = pow(theta, -2.0 * (double)i / (double)D);
  const double a = (double)pos * inv;
  tab[idx] = make_float2((float)cos(a), (float)sin(a));
}

__global__ void k_read_kv(KVGeom kv, int layer, int slot, int pos0, int n, float* k_out, float* v_out) {
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const int D = kv.D, hkv = kv.hkv;
  if (idx >= (long long)n * hkv * D) return;
  const int d = (int)(idx % D);
  const int h = (int)((idx / D) % hkv);
  const int t = (int)(idx / ((long long)D * hkv));
  const int pos = pos0 + t;
  const int pi = pos >> 6;
  int pg = pi < kv.max_pages_per_slot ? kv.page_table[(size_t)slot * kv.max_pages_per_slot + pi] : -1;
  if (pg < 0 || pg >= kv.max_pages) {
    k_out[idx] = 0.f;
    v_out[idx] = 0.f;
    return;
  }
  const size_t blk = (size_t)layer * kv.layer_stride + ((size_t)pg * hkv + h) * (64 * D);
  k_out[idx] = __half2float(kv.k_pool[blk + k_swz(pos & 63, d)]);
  v_out[idx] = __half2float(kv.v_pool[blk + v_swz(d, pos & 63)]);
}

__global__ void k_slot_lengths(const int* slots, int batch, const int* ctx_len, int max_slots, int* out) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= batch) return;
  const int s = slots[b];
  out[b] = (s >= 0 && s < max_slots) ? ctx_len[s] : -1;
}

// The stand-in verify's work (see k_harness_verify).
DFL_DEV void verify_body(const int* slots, int batch, int S, const int* draft, const int* match, const int* offs,
                         int rounds_cap, int* round_ctr, int* target, int vocab, const bf16* feat_stream,
                         int stream_rows, bf16* feats_out, int F, const int* ctx_len, int max_slots) {
  if (blockIdx.x == 0) {
    const int r = *round_ctr;
    const int rr = r % rounds_cap;
    for (int idx = threadIdx.x; idx < batch * S; idx += blockDim.x) {
      const int b = idx / S, i = idx % S;
      const size_t o = ((size_t)rr * batch + b) * S + i;
      const int u = offs[o];
      int t;
      if (i < S - 1) {
        const int d = draft[b * (S - 1) + i];
        t = match[o] ? d : (u == d ? (u + 1) % vocab : u);
      } else {
        t = u;
      }
      target[idx] = t;
    }
    __syncthreads();
    if (threadIdx.x == 0) *round_ctr = r + 1;
    return;
  }
  const int row = blockIdx.x - 1;
  const int b = row / S, i = row % S;
  const int slot = slots[b];
  if (slot < 0 || slot >= max_slots) return;
  int pos = ctx_len[slot] + i;
  if (pos >= stream_rows) pos = stream_rows - 1;
  const uint4* src = reinterpret_cast<const uint4*>(feat_stream + ((size_t)b * stream_rows + pos) * F);
  uint4* dst = reinterpret_cast<uint4*>(feats_out + (size_t)row * F);
  for (int k = threadIdx.x; k < F / 8; k += blockDim.x) dst[k] = src[k];
}

// Benchmark stand-in for the target's verify (not part of the method).
// Block 0 builds the target tokens of round (*round_ctr)++; blocks 1.. copy
// the target features of the S block positions from a position-indexed stream.
// With `stamp` non-null, stamp[0] receives %globaltimer when the kernel may
// start its work (the drafter's last kernel complete) and stamp[1] when its
// last block is done (counted on blocks_done, left at zero).
__global__ void k_harness_verify(const int* slots, int batch, int S, const int* draft, const int* match, const int* offs,
                                 int rounds_cap, int* round_ctr, int* target, int vocab,
                                 const bf16* feat_stream, int stream_rows, bf16* feats_out, int F,
                                 const int* ctx_len, int max_slots, unsigned long long* stamp,
                                 unsigned* blocks_done) {
  pdl_launch_dependents();
  pdl_wait();
  if (stamp && blockIdx.x == 0 && threadIdx.x == 0) stamp[0] = globaltimer();
  verify_body(slots, batch, S, draft, match, offs, rounds_cap, round_ctr, target, vocab, feat_stream, stream_rows,
              feats_out, F, ctx_len, max_slots);
  if (stamp) {
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      if (atomicAdd(blocks_done, 1u) == gridDim.x - 1) {
        stamp[1] = globaltimer();
        *blocks_done = 0u;
      }
    }
  }
}

// Failure-detection check: thread 0 waits on an mbarrier nothing arrives at,
// with a short limit, through the pipelines' own bounded wait; it gives up,
// sets DFLASH_DEV_TIMEOUT and returns.  A second wait after the give-up
// returns at once (the aborted flag), as the pipelines' drain paths rely on.
__global__ void k_wait_check(uint32_t* status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    bool aborted = false;
    mbar_wait_for(&bar, 0, status, &aborted, limit_ns);
    mbar_wait_for(&bar, 0, status, &aborted, limit_ns);
  }
}

__global__ void k_tap(const float* __restrict__ h, int H, bf16* __restrict__ feats, int tap, int n_fused) {
  pdl_launch_dependents();
  pdl_wait();
  const int row = blockIdx.x;
  const float* src = h + (size_t)row * H;
  bf16* dst = feats + ((size_t)row * n_fused + tap) * H;
  for (int k = threadIdx.x; k < H; k += blockDim.x) dst[k] = __float2bfloat16_rn(src[k]);
}

}  // namespace

cudaError_t launch_wait_check(uint32_t* status, unsigned long long limit_ns, cudaStream_t s) {
  k_wait_check<<<1, 32, 0, s>>>(status, limit_ns);
  return cudaGetLastError();
}

cudaError_t launch_tap(const float* h, int M, int H, bf16* feats, int tap, int n_fused, cudaStream_t s) {
  cudaLaunchAttribute a[1];
  cudaLaunchConfig_t c = cfg_of(dim3(M), dim3(256), s, a);
  return cudaLaunchKernelEx(&c, k_tap, h, H, feats, tap, n_fused);
}

cudaError_t launch_pack_weight(const bf16* src, void* dst, int N, int K, int n_tiles, int swiglu_I, bool to_f16,
                               uint32_t* status, cudaStream_t s) {
  const long long total = (long long)n_tiles * (K / 64) * 128 * 8;
  const long long blocks = std::min<long long>((total + 255) / 256, 1LL << 20);
  k_pack_weight<<<(unsigned)blocks, 256, 0, s>>>(src, static_cast<uint16_t*>(dst), N, K, n_tiles, swiglu_I,
                                                 to_f16 ? 1 : 0, status);
  return cudaGetLastError();
}

cudaError_t launch_pack_weight_fp8(const bf16* src, uint8_t* dst, float* scale, int N, int K, int n_tiles,
                                   int swiglu_I, cudaStream_t s) {
  const int rows = n_tiles * 128;
  k_fp8_scale<<<(rows * 32 + 255) / 256, 256, 0, s>>>(src, scale, N, K, rows, swiglu_I);
  cudaError_t e = cudaGetLastError();
  if (e) return e;
  const long long total = (long long)n_tiles * (K / 64) * 128 * 4;
  const long long blocks = std::min<long long>((total + 255) / 256, 1LL << 20);
  k_pack_fp8<<<(unsigned)blocks, 256, 0, s>>>(src, scale, dst, N, K, n_tiles, swiglu_I);
  return cudaGetLastError();
}

cudaError_t launch_gain_f32(const bf16* src, float* dst, int n, cudaStream_t s) {
  k_gain_f32<<<(n + 255) / 256, 256, 0, s>>>(src, dst, n);
  return cudaGetLastError();
}

cudaError_t launch_embed(const int* slots, int batch, const int* last_tok, int mask_id, int vocab,
                         const void* embed_pk, const float* embed_scale, const float* gain, int H, float* h, f16* hg,
                         float* ss, unsigned long long* keys, const BlockCtx& bc, uint32_t* status, cudaStream_t s) {
  cudaLaunchAttribute a[1];
  const int M = batch * DFL_BLOCK;
  int threads = (H / 128) * 32;
  if (threads > 1024) threads = 1024;
  cudaLaunchConfig_t c = cfg_of(dim3(M), dim3(threads), s, a);
  return cudaLaunchKernelEx(&c, k_embed, slots, last_tok, mask_id, vocab, embed_pk, embed_scale, gain, H, M, h, hg,
                            ss, keys, bc, status);
}

cudaError_t launch_page_alloc(const int* slots, int batch, int S, const int* n_new, int rows_per_req, int* ctx_len,
                              int* pos0, int* n_pages, int* page_table, int mpps, int* free_stack, int* free_top,
                              int* n_eff, int* slots_ok, int max_slots, uint32_t* status, cudaStream_t s,
                              int* row_off, int* n_live) {
  cudaLaunchAttribute a[1];
  cudaLaunchConfig_t c = cfg_of(dim3(1), dim3(32), s, a);
  return cudaLaunchKernelEx(&c, k_page_alloc, slots, batch, S, n_new, rows_per_req, ctx_len, pos0, n_pages,
                            page_table, mpps, free_stack, free_top, n_eff, slots_ok, max_slots, status, row_off,
                            n_live);
}

cudaError_t launch_compact_rows(const bf16* feats, int batch, int rows_per_req, int F, const int* n_eff,
                                const int* row_off, bf16* dst, int* row_map, cudaStream_t s) {
  cudaLaunchAttribute a[1];
  cudaLaunchConfig_t c = cfg_of(dim3((unsigned)rows_per_req, (unsigned)batch), dim3(256), s, a);
  return cudaLaunchKernelEx(&c, k_compact_rows, feats, rows_per_req, F, n_eff, row_off, dst, row_map);
}

cudaError_t launch_accept(const int* slots, int batch, int S, const int* draft, const int* target, int* accept_len,
                          int* bonus, int* ctx_out, int* ctx_len, int max_slots, uint32_t* status,
                          cudaStream_t s) {
  cudaLaunchAttribute a[1];
  cudaLaunchConfig_t c = cfg_of(dim3((batch + 3) / 4), dim3(128), s, a);
  return cudaLaunchKernelEx(&c, k_accept, slots, batch, S, draft, target, accept_len, bonus, ctx_out,
                            (const int*)ctx_len, max_slots, status);
}

cudaError_t launch_reset_slot(int slot, int* ctx_len, int* n_pages, int* page_table, int mpps, int* free_stack,
                              int* free_top, cudaStream_t s) {
  cudaLaunchAttribute a[1];
  cudaLaunchConfig_t c = cfg_of(dim3(1), dim3(32), s, a);
  return cudaLaunchKernelEx(&c, k_reset_slot, slot, ctx_len, n_pages, page_table, mpps, free_stack, free_top);
}

cudaError_t launch_pool_init(int* free_stack, int* free_top, int max_pages, cudaStream_t s) {
  k_pool_init<<<(max_pages + 255) / 256, 256, 0, s>>>(free_stack, free_top, max_pages);
  return cudaGetLastError();
}

cudaError_t launch_rope_table(float2* tab, int max_pos, int D, float theta, cudaStream_t s) {
  const long long n = (long long)max_pos * (D / 2);
  k_rope_table<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(tab, max_pos, D, (double)theta);
  return cudaGetLastError();
}

cudaError_t launch_read_kv(const KVGeom& kv, int layer, int slot, int pos0, int n, float* k_out, float* v_out,
                           cudaStream_t s) {
  const long long tot = (long long)n * kv.hkv * kv.D;
  if (tot == 0) return cudaSuccess;
  k_read_kv<<<(unsigned)((tot + 255) / 256), 256, 0, s>>>(kv, layer, slot, pos0, n, k_out, v_out);
  return cudaGetLastError();
}

cudaError_t launch_slot_lengths(const int* slots, int batch, const int* ctx_len, int max_slots, int* out,
                                cudaStream_t s) {
  k_slot_lengths<<<(batch + 127) / 128, 128, 0, s>>>(slots, batch, ctx_len, max_slots, out);
  return cudaGetLastError();
}

cudaError_t launch_harness_verify(const int* slots, int batch, int S, const int* draft, const int* match,
                                  const int* offs, int rounds_cap, int* round_ctr, int* target, int vocab,
                                  const bf16* feat_stream, int stream_rows, bf16* feats_out, int F, const int* ctx_len,
                                  int max_slots, unsigned long long* stamp, unsigned* blocks_done, cudaStream_t s) {
  cudaLaunchAttribute a[1];
  const int blocks = 1 + (feat_stream ? batch * S : 0);
  cudaLaunchConfig_t c = cfg_of(dim3(blocks), dim3(256), s, a);
  return cudaLaunchKernelEx(&c, k_harness_verify, slots, batch, S, draft, match, offs, rounds_cap, round_ctr, target,
                            vocab, feat_stream, stream_rows, feats_out, F, ctx_len, max_slots, stamp, blocks_done);
}
