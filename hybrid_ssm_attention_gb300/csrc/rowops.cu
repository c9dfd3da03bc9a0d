// Row kernels of the verify step and the accept / commit kernels.
//
//  embed_norm     X[t] = E[token_t]; xn[t] = RMSNorm(X[t]) in storage dtype
//  residual_norm  X[t] += (GEMM partials)[t]; xn[t] = RMSNorm(X[t])
//  mlp_act        h[t][j] = silu(gate) * up from the gate/up GEMM partials
//  logits         logits[t][j] = head GEMM partials
//  probs          temperature / top-k softmax of each logits row (model card,
//                 "Library" example: T = 1.0, top_k = 4)
//  accept         the exact accept rule of speculative sampling (EvSpark
//                 preprint abstract; discussion post, "What we implemented"):
//                 greedy match or u*q < p, residual / bonus resampling
//  commit         per-position state slicing by bank flips (abstract, (i))
//
// Reductions run in a fixed order (per-thread strided partials, then a
// butterfly), so results are reproducible and independent of the block size.
#include <cooperative_groups.h>

#include "evs_internal.cuh"

namespace cg = cooperative_groups;

namespace evs {
namespace {

template <typename V, typename Op>
__device__ V block_reduce(V v, Op op, V* scratch /* >= 32 */) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = op(v, __shfl_xor_sync(0xffffffffu, v, o));
  __syncthreads();
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  V r = scratch[0];
  for (int w = 1; w < nw; ++w) r = op(r, scratch[w]);
  __syncthreads();
  return r;
}

struct AddF { __device__ float operator()(float a, float b) const { return a + b; } };
struct MaxF { __device__ float operator()(float a, float b) const { return fmaxf(a, b); } };
struct AddU { __device__ unsigned long long operator()(unsigned long long a, unsigned long long b) const { return a + b; } };

// Embedding + RMSNorm of one token row, spread over the CTAs of a
// thread-block cluster (grid (CL, n), cluster (CL, 1, 1)): CTA r owns
// columns [r*d/CL, (r+1)*d/CL).  Sets X[t] = E[token_t], marks the block
// pending, writes xn[t].  Each CTA's sum of squares is summed over the
// cluster's shared memory in rank order, so the result does not depend on
// the number of rows.
template <typename T>
__global__ void __launch_bounds__(256) embed_norm_kernel(const T* E, const int32_t* tokens, int V, float* X,
                                                         int d, float eps, T* xn, const __grid_constant__ SeqRows sr,
                                                         const __grid_constant__ SeqPtrs<evs_book*> books) {
  __shared__ float scratch[32];
  __shared__ float ss_cta;
  cg::cluster_group cl = cg::this_cluster();
  const int ncl = (int)cl.num_blocks(), rank = (int)cl.block_rank();
  const int t = blockIdx.y;
  const int cols = d / ncl, c0 = rank * cols;
  pdl_trigger();
  pdl_wait();
  float* x = X + (size_t)t * d;
  float ss = 0.f;
  // row t belongs to sequence sq; its first row records the block length
  const int sq = seq_of_row(sr, t);
  evs_book* book = books.p[sq];
  if (t == sr.row0[sq] && rank == 0 && threadIdx.x == 0) book->pending_n = sr.row0[sq + 1] - sr.row0[sq];
  const int tok = tokens[t];
  const bool ok = tok >= 0 && tok < V;
  if (!ok && rank == 0 && threadIdx.x == 0) set_status(book, EVS_DEV_BAD_TOKEN);
  for (int c = c0 + threadIdx.x; c < c0 + cols; c += blockDim.x) {
    const float v = ok ? to_f(E[(size_t)tok * d + c]) : 0.f;
    x[c] = v;
    ss = fmaf(v, v, ss);
  }
  ss = block_reduce(ss, AddF(), scratch);
  if (threadIdx.x == 0) ss_cta = ss;
  cl.sync();
  float tot = 0.f;
  for (int q = 0; q < ncl; ++q) tot += *cl.map_shared_rank(&ss_cta, q);
  const float den = sqrtf(tot / (float)d + eps), rden = 1.f / den;
  T* xo = xn + (size_t)t * d;
  for (int c = c0 + threadIdx.x; c < c0 + cols; c += blockDim.x) xo[c] = from_f<T>(div_row(x[c], den, rden));
  cl.sync();  // ss_cta stays alive until every CTA of the cluster has read it
}

// CTAs per token row: up to 8, each owning >= 256 columns (a multiple of 32)
int row_cluster(int d) {
  int cl = 8;
  while (cl > 1 && (d % (cl * 32) != 0 || d / cl < 256)) cl >>= 1;
  return cl;
}

// RMSNorm of rows whose residual update the out / down GEMM already applied:
// the row's sum of squares is the GEMM's per-tile sums added in tile order.
template <typename T>
__global__ void __launch_bounds__(256) norm_apply_kernel(const float* X, const float* ss, int ntiles, int d,
                                                         float eps, T* xn) {
  __shared__ float s_den, s_rcp;
  const int t = blockIdx.y;
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  pdl_trigger();
  pdl_wait();
  // this thread's residual value is loaded alongside the per-tile sums
  const float x = c < d ? __ldcg(X + (size_t)t * d + c) : 0.f;
  if (threadIdx.x < 32) {
    // the per-tile sums, 32 loads in flight at a time, added in tile order
    const int lane = threadIdx.x;
    float tot = 0.f;
    for (int k0 = 0; k0 < ntiles; k0 += 32) {
      const float mine = k0 + lane < ntiles ? __ldcg(ss + (k0 + lane) * ROWS_MAX + t) : 0.f;
      for (int j = 0; j < 32 && k0 + j < ntiles; ++j) tot += __shfl_sync(0xffffffffu, mine, j);
    }
    if (lane == 0) {
      s_den = sqrtf(tot / (float)d + eps);
      s_rcp = 1.f / s_den;
    }
  }
  __syncthreads();
  if (c < d) xn[(size_t)t * d + c] = from_f<T>(div_row(x, s_den, s_rcp));
}

// Residual add and RMSNorm of rows whose out / down GEMM left partial slots.
// A cluster of ncl CTAs per row; warp w of CTA r owns 128-column tile
// r * warps + w, lane l its four columns 4l .. 4l+3 (float4 loads of the
// residual row and of every slot).  The tile's sum of squares follows the
// GEMM_RESID epilogue exactly: there, column c sits in lane c % 32 of warp
// c / 32 and each warp's squares meet by xor butterfly over 16, 8, 4, 2, 1,
// then the four warps are added in order.  Here the xor partners c ^ 16,
// c ^ 8, c ^ 4 are lanes l ^ 4, l ^ 2, l ^ 1 and c ^ 2, c ^ 1 are within
// the lane; with commuted operands every partial sum is the same value,
// so the tile sum is bit-identical.  The row's sum adds the tile sums in
// tile order; each CTA pushes its tile sums into every CTA's shared memory
// before the one cluster barrier, after which only local memory is read.
template <typename T>
__global__ void __launch_bounds__(256) resid_norm_kernel(float* X, const __grid_constant__ SrcSlots src, int d,
                                                         float eps, T* xn) {
  __shared__ float s_all[RESID_TILES_ROW];  // the row's tile sums, tile order
  __shared__ float s_den, s_rcp;
  cg::cluster_group cl = cg::this_cluster();
  const int ncl = (int)cl.num_blocks(), rank = (int)cl.block_rank();
  const int t = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = rank * (blockDim.x >> 5) + warp, ntiles = d / TILE_M;
  const int col = tile * TILE_M + 4 * lane;
  pdl_trigger();
  const SrcSlots::Col c = src.at(col);
  pdl_wait();
  float* xr = X + (size_t)t * d + col;
  const size_t stride = (size_t)src.rows * TILE_M;
  const float* p = c.p + (size_t)t * TILE_M;
  // every load first (X may alias the slots for all the compiler knows):
  // the row, then all of the tile's slots (at most SLOTS_RESID_MAX, checked
  // on the host) without a branch
  float4 x = __ldcg(reinterpret_cast<const float4*>(xr));
  const float4 v0 = __ldcg(reinterpret_cast<const float4*>(p));
  float4 a[SLOTS_RESID_MAX];
#pragma unroll
  for (int j = 1; j < SLOTS_RESID_MAX; ++j)
    a[j] = c.cnt > j ? __ldcg(reinterpret_cast<const float4*>(p + j * stride)) : make_float4(0.f, 0.f, 0.f, 0.f);
  float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int j = 1; j < SLOTS_RESID_MAX; ++j) v.x += a[j].x, v.y += a[j].y, v.z += a[j].z, v.w += a[j].w;
  x.x += v0.x + v.x;
  x.y += v0.y + v.y;
  x.z += v0.z + v.z;
  x.w += v0.w + v.w;
  *reinterpret_cast<float4*>(xr) = x;
  float q[4] = {x.x * x.x, x.y * x.y, x.z * x.z, x.w * x.w};
#pragma unroll
  for (int o = 4; o > 0; o >>= 1)  // column xor 16, 8, 4
#pragma unroll
    for (int k = 0; k < 4; ++k) q[k] += __shfl_xor_sync(0xffffffffu, q[k], o);
  const float wsum = (q[0] + q[2]) + (q[1] + q[3]);  // column xor 2, then 1
  // tile sum: the four 32-column warps of the epilogue (lanes 0, 8, 16, 24)
  const float w1 = __shfl_sync(0xffffffffu, wsum, 8), w2 = __shfl_sync(0xffffffffu, wsum, 16);
  const float w3 = __shfl_sync(0xffffffffu, wsum, 24);
  const float ts = ((wsum + w1) + w2) + w3;
  if (lane < ncl) *cl.map_shared_rank(&s_all[tile], lane) = ts;
  cl.sync();
  if (warp == 0) {
    // the tile sums, 32 at a time, added in tile order
    float tot = 0.f;
    for (int q0 = 0; q0 < ntiles; q0 += 32) {
      const float mine = q0 + lane < ntiles ? s_all[q0 + lane] : 0.f;
      for (int k = 0; k < 32 && q0 + k < ntiles; ++k) tot += __shfl_sync(0xffffffffu, mine, k);
    }
    if (lane == 0) {
      s_den = sqrtf(tot / (float)d + eps);
      s_rcp = 1.f / s_den;
    }
  }
  __syncthreads();
  const float den = s_den, rden = s_rcp;
  T* xo = xn + (size_t)t * d + col;
  xo[0] = from_f<T>(div_row(x.x, den, rden));
  xo[1] = from_f<T>(div_row(x.y, den, rden));
  xo[2] = from_f<T>(div_row(x.z, den, rden));
  xo[3] = from_f<T>(div_row(x.w, den, rden));
}

// CTAs per row: the fewest of 1, 2, 4, 8 that leave <= 8 whole tiles (one
// per warp) to each; 0 if none fits
int resid_cluster(int d) {
  if (d % TILE_M) return 0;
  const int nt = d / TILE_M;
  for (int cl = 1; cl <= 8; cl <<= 1)
    if (nt % cl == 0 && nt / cl <= 8) return cl;
  return 0;
}

template <typename T, typename Src>
__global__ void mlp_act_kernel(const __grid_constant__ Src gu, int F, int il, T* h) {
  const int t = blockIdx.y, j = blockIdx.x * blockDim.x + threadIdx.x;
  pdl_trigger();
  const int gj = il ? (j / 64) * 128 + j % 64 : j, uj = il ? gj + 64 : F + j;
  typename Src::Col cg{}, cu{};
  if (j < F) cg = gu.at(gj), cu = gu.at(uj);
  pdl_wait();
  if (j >= F) return;
  const float gt = gu.get(cg, t, gj), up = gu.get(cu, t, uj);
  h[(size_t)t * F + j] = from_f<T>(silu_f(gt) * up);
}

// Orderable key of a float: a larger value has a larger key; -0 and +0
// share one key (they compare equal); NaN has key 0, below every number, so
// a NaN enters a top-k support only when fewer than k numbers exist (the
// oracle's stable descending sort puts NaN last).
__device__ __forceinline__ unsigned int ord_key(float x) {
  if (x != x) return 0u;
  if (x == 0.f) x = 0.f;
  const unsigned int b = __float_as_uint(x);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Inclusive prefix sum of v over the block in thread order (blockDim.x a
// multiple of 32, at most 1024); scratch >= 32 ints.
__device__ int block_scan_incl(int v, int* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += y;
  }
  if (lane == 31) scratch[warp] = v;
  __syncthreads();
  int base = 0;
  for (int w = 0; w < warp; ++w) base += scratch[w];
  __syncthreads();
  return v + base;
}

// Shared scratch of row_topk_softmax.
struct TopkScratch {
  float f[32];
  int i[32];
  unsigned int hist[256];
  unsigned int prefix;
  int remain, eq;
};

// Top-k softmax of the row l_s[V] (shared memory, written and synchronised
// by the caller) by the whole block: w_s[j] = p_j.  The k-th largest logit
// is found by radix select over the four bytes of its orderable key (a
// 256-bin histogram per byte, O(V) work); entries above it are kept, and of
// the entries equal to it the lowest-indexed ones fill the remaining places
// (ties to the lower index).  k <= 0 or k >= V keeps every entry.
__device__ void row_topk_softmax(const float* l_s, float* w_s, int V, float T, int k, TopkScratch& ts) {
  const int tid = threadIdx.x, nth = blockDim.x;
  const bool use_k = k > 0 && k < V;
  unsigned int kth = 0;  // key of the k-th largest entry
  int need_eq = 0, n_eq = 0;
  if (use_k) {
    unsigned int prefix = 0, mask = 0;
    int remain = k;
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int i = tid; i < 256; i += nth) ts.hist[i] = 0;
      __syncthreads();
      for (int j = tid; j < V; j += nth) {
        const unsigned int key = ord_key(l_s[j]);
        if ((key & mask) == prefix) atomicAdd(&ts.hist[(key >> shift) & 255u], 1u);
      }
      __syncthreads();
      if (tid < 32) {
        // the digit D holding the remain-th largest of the entries matching
        // prefix: count(bins > D) < remain <= count(bins >= D).  Lane l owns
        // bins 8l .. 8l+7; a suffix sum over the lanes finds the one lane
        // whose bins hold D, which scans its eight bins from the top.
        const int lane = tid;
        int c[8], tot = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) tot += c[e] = (int)ts.hist[8 * lane + e];
        int suf = tot;  // bins of lanes >= lane
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_down_sync(0xffffffffu, suf, o);
          if (lane + o < 32) suf += y;
        }
        int acc = suf - tot;  // bins of lanes above this one
        if (acc < remain && remain <= acc + tot) {
          int D = 8 * lane, eq = c[0];
#pragma unroll
          for (int e = 7; e >= 0; --e) {
            if (acc + c[e] >= remain) {
              D = 8 * lane + e;
              eq = c[e];
              break;
            }
            acc += c[e];
          }
          ts.prefix = prefix | ((unsigned int)D << shift);
          ts.remain = remain - acc;
          ts.eq = eq;
        }
      }
      __syncthreads();
      prefix = ts.prefix;
      remain = ts.remain;
      mask |= 255u << shift;
      __syncthreads();
    }
    kth = prefix;
    need_eq = remain;  // entries equal to kth to keep (k - remain entries lie above it)
    n_eq = ts.eq;      // entries equal to kth in all
  }
  float mx = -INFINITY;
  if (!use_k || need_eq == n_eq) {
    // no tie straddles the cut: keep every entry at or above the k-th key
    for (int j = tid; j < V; j += nth) {
      const bool keep = !use_k || ord_key(l_s[j]) >= kth;
      w_s[j] = keep ? 1.f : 0.f;
      if (keep) mx = fmaxf(mx, l_s[j]);
    }
  } else {
    // ties at the cut: rank the equal entries by index (thread i owns the
    // contiguous index range [i*seg, (i+1)*seg), ranks by a block scan)
    const int seg = (V + nth - 1) / nth;
    const int j0 = min(V, tid * seg), j1 = min(V, j0 + seg);
    int c = 0;
    for (int j = j0; j < j1; ++j) c += ord_key(l_s[j]) == kth;
    int rank = block_scan_incl(c, ts.i) - c;  // equal entries before this range
    for (int j = j0; j < j1; ++j) {
      const unsigned int key = ord_key(l_s[j]);
      bool keep = key > kth;
      if (key == kth) keep = rank++ < need_eq;
      w_s[j] = keep ? 1.f : 0.f;
      if (keep) mx = fmaxf(mx, l_s[j]);
    }
  }
  mx = block_reduce(mx, MaxF(), ts.f);
  float sum = 0.f;
  for (int j = tid; j < V; j += nth) {
    const float w = w_s[j] != 0.f ? expf((l_s[j] - mx) / T) : 0.f;
    w_s[j] = w;
    sum += w;
  }
  sum = block_reduce(sum, AddF(), ts.f);
  for (int j = tid; j < V; j += nth) w_s[j] = w_s[j] / sum;
  __syncthreads();
}

// One CTA per row: the target distribution (temperature, top-k).
__global__ void __launch_bounds__(256) probs_kernel(const float* logits, int V, float T, int k, float* p) {
  extern __shared__ float sm[];
  __shared__ TopkScratch ts;
  float* l_s = sm;        // [V]
  float* w_s = sm + V;    // [V]
  const int t = blockIdx.x;
  pdl_trigger();
  pdl_wait();
  for (int j = threadIdx.x; j < V; j += blockDim.x) l_s[j] = logits[(size_t)t * V + j];
  __syncthreads();
  row_topk_softmax(l_s, w_s, V, T, k, ts);
  for (int j = threadIdx.x; j < V; j += blockDim.x) p[(size_t)t * V + j] = w_s[j];
}

// argmax over a row by one warp, same ties rule (lowest index); all-NaN -> 0
__device__ int warp_argmax(const float* row, int V) {
  const int lane = threadIdx.x & 31;
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  for (int j = lane; j < V; j += 32) {
    const float v = row[j];
    if (v > bv || (v == bv && j < bi)) { bv = v; bi = j; }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
  }
  return bi == 0x7fffffff ? 0 : bi;
}

__device__ __forceinline__ unsigned int ladder_weight(float w) {
  // floor(w * 2^24): the scaling is exact in float32, the conversion truncates
  return (unsigned int)(fmaxf(w, 0.f) * 16777216.0f);
}

// Inverse CDF on integer weights: smallest j with prefix_j > thr.
// Thread i owns the contiguous slice [i*seg, (i+1)*seg).
__device__ int ladder_find(const unsigned int* W, int V, unsigned long long thr, unsigned long long* us,
                           int* found) {
  const int seg = (V + blockDim.x - 1) / blockDim.x;
  const int j0 = min(V, (int)threadIdx.x * seg), j1 = min(V, j0 + seg);
  unsigned long long local = 0;
  for (int j = j0; j < j1; ++j) local += W[j];
  // exclusive scan of the per-thread sums, in thread order
  us[threadIdx.x] = local;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long run = 0;
    for (int i = 0; i < (int)blockDim.x; ++i) {
      const unsigned long long x = us[i];
      us[i] = run;
      run += x;
    }
    *found = -1;
  }
  __syncthreads();
  unsigned long long pre = us[threadIdx.x];
  if (pre <= thr && thr < pre + local) {
    for (int j = j0; j < j1; ++j) {
      pre += W[j];
      if (pre > thr) { *found = j; break; }
    }
  }
  __syncthreads();
  return *found;
}

__device__ void commit_one(evs_book* book, int keep, int n_explicit) {
  const int n = n_explicit > 0 ? n_explicit : book->pending_n;
  if (n <= 0 || keep < 0 || keep > n) {
    set_status(book, EVS_DEV_BAD_KEEP);
    book->pending_n = 0;
    return;
  }
  // FIR windows follow pos (ring rows by absolute position)
  if (keep > 0) {
    book->iir_bank ^= 1;
    book->iir_slot = keep - 1;
  }
  book->pos += keep;
  book->pending_n = 0;
}

// One CTA per sequence b of sr: its rows r0 = sr.row0[b] .. + n - 1 of p,
// q, drafts and u (row r0 + i of q / drafts: draft i + 1); results to
// out_a[b], out_tok[b].
// books.p[b] (may be null): sequence b's bookkeeping, whose status gets
// EVS_DEV_BAD_PROBS when a sampled row has no integer mass.
__global__ void __launch_bounds__(256) accept_kernel(const float* p, const float* q, const int32_t* drafts,
                                                     const float* u, const __grid_constant__ SeqRows sr, int V,
                                                     int mode, int32_t* out_a, int32_t* out_tok,
                                                     const __grid_constant__ SeqPtrs<evs_book*> books, int commit) {
  extern __shared__ unsigned int Wsm[];  // [V], then s_arg[n], s_ok[n]
  __shared__ unsigned long long us[256];
  __shared__ int found;
  const int b = blockIdx.x, r0 = sr.row0[b], n = sr.row0[b + 1] - r0;
  p += (size_t)r0 * V;
  if (q) q += (size_t)r0 * V;
  if (drafts) drafts += r0;
  if (u) u += r0;
  out_a += b;
  out_tok += b;
  int* s_arg = reinterpret_cast<int*>(Wsm + V);  // greedy: argmax of every row
  int* s_ok = s_arg + n;                          // [i]: draft i passes its own test (1..gamma)
  pdl_trigger();
  pdl_wait();
  const int gamma = n - 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  // every row's test at once (one warp per row), then the first rejection
  if (mode == EVS_GREEDY) {
    for (int r = warp; r < n; r += nw) {
      const int am = warp_argmax(p + (size_t)r * V, V);
      if (lane == 0) s_arg[r] = am;
    }
    __syncthreads();
    for (int i = 1 + threadIdx.x; i <= gamma; i += blockDim.x) s_ok[i] = drafts[i - 1] == s_arg[i - 1];
  } else {
    for (int i = 1 + threadIdx.x; i <= gamma; i += blockDim.x) {
      const int d = drafts[i - 1];
      s_ok[i] = d >= 0 && d < V && __fmul_rn(u[i - 1], q[(size_t)(i - 1) * V + d]) < p[(size_t)(i - 1) * V + d];
    }
  }
  __syncthreads();
  int a = gamma;
  for (int i = 1; i <= gamma; ++i)
    if (!s_ok[i]) { a = i - 1; break; }
  int token;
  if (mode == EVS_GREEDY) {
    token = s_arg[a];
  } else {
    const float* pa = p + (size_t)a * V;
    unsigned long long S = 0;
    if (a < gamma) {
      const float* qa = q + (size_t)a * V;
      unsigned long long loc = 0;
      for (int j = threadIdx.x; j < V; j += blockDim.x) {
        Wsm[j] = ladder_weight(__fsub_rn(pa[j], qa[j]));
        loc += Wsm[j];
      }
      S = block_reduce(loc, AddU(), us);
    }
    if (S == 0) {
      unsigned long long loc = 0;
      for (int j = threadIdx.x; j < V; j += blockDim.x) {
        Wsm[j] = ladder_weight(pa[j]);
        loc += Wsm[j];
      }
      S = block_reduce(loc, AddU(), us);
    }
    __syncthreads();
    // floor(u 2^24), held below 2^24 so that u = 1 (outside [0, 1)) still
    // lands on the last entry with mass
    const unsigned long long U =
        min((unsigned long long)(unsigned int)(u[gamma] * 16777216.0f), 16777215ull);
    const unsigned long long thr = (U * S) >> 24;
    token = ladder_find(Wsm, V, thr, us, &found);
    __syncthreads();  // every thread has read found before it is reused
    if (token < 0) {
      // neither the residual nor p_a has integer mass (a NaN or all-zero
      // row): the row's argmax stands in, and the state is flagged
      if (warp == 0) {
        const int am = warp_argmax(pa, V);
        if (lane == 0) found = am;
      }
      __syncthreads();
      token = found;
      if (threadIdx.x == 0 && books.p[b]) set_status(books.p[b], EVS_DEV_BAD_PROBS);
    }
  }
  if (threadIdx.x == 0) {
    out_a[0] = a;
    out_tok[0] = token;
    // a round's commit with keep = a + 1, here instead of one more launch
    if (commit && books.p[b]) commit_one(books.p[b], a + 1, 0);
  }
}

// Drafter-side Markov head (preprint abstract, contribution (ii); model
// card, drafter description): the gamma drafts are drawn one after another in
// one CTA.  Slot i's logits are the trunk's row i plus row prev of the V x V
// Markov matrix, prev being the pending token for the first slot and the
// previous draft after it; q_i is their top-k softmax at temperature T and
// the draft is q_i's integer-ladder sample with uniform u[i] (greedy: the
// argmax of the logits, lowest index on ties).  A pending token outside
// [0, V) selects row 0.
__global__ void __launch_bounds__(256) markov_draft_kernel(const float* trunk, const float* M, int V,
                                                           const int32_t* prev_dev, const float* u, int gamma,
                                                           float T, int k, int mode, int32_t* drafts, float* q) {
  extern __shared__ float sm[];
  __shared__ TopkScratch ts;
  __shared__ unsigned long long us[256];
  __shared__ int found;
  float* l_s = sm;                                           // [V] logits of the slot
  float* w_s = sm + V;                                       // [V] q of the slot
  unsigned int* Wl = reinterpret_cast<unsigned int*>(sm + 2 * V);  // [V] ladder weights
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_trigger();
  pdl_wait();
  int prev = prev_dev[0];
  if (prev < 0 || prev >= V) prev = 0;
  for (int i = 0; i < gamma; ++i) {
    const float* mr = M + (size_t)prev * V;
    const float* tr = trunk + (size_t)i * V;
    for (int j = threadIdx.x; j < V; j += blockDim.x) l_s[j] = __fadd_rn(tr[j], mr[j]);
    __syncthreads();
    row_topk_softmax(l_s, w_s, V, T, k, ts);
    for (int j = threadIdx.x; j < V; j += blockDim.x) q[(size_t)i * V + j] = w_s[j];
    int d = -1;
    if (mode == EVS_SAMPLE) {
      unsigned long long loc = 0;
      for (int j = threadIdx.x; j < V; j += blockDim.x) {
        Wl[j] = ladder_weight(w_s[j]);
        loc += Wl[j];
      }
      const unsigned long long S = block_reduce(loc, AddU(), us);
      __syncthreads();
      const unsigned long long U = min((unsigned long long)(unsigned int)(u[i] * 16777216.0f), 16777215ull);
      d = ladder_find(Wl, V, (U * S) >> 24, us, &found);
      __syncthreads();  // every thread has read found before it is reused
    }
    if (d < 0) {  // greedy, or a row without integer mass
      if (warp == 0) {
        const int am = warp_argmax(l_s, V);
        if (lane == 0) found = am;
      }
      __syncthreads();
      d = found;
    }
    if (threadIdx.x == 0) drafts[i] = d;
    prev = d;
    __syncthreads();  // every thread has read found and l_s before the next slot
  }
}

// The same draft chain for 0 < top_k <= 8 and V <= 8192, with the support
// found by merging sorted lists instead of a radix select.  Order: larger
// logit first, lower index on ties (the oracle's stable order; a NaN never
// enters).  Each of the 256 threads keeps the best KM of its strided entries
// j = tid + 256 e in registers; a butterfly over the warp merges the lists of
// lane pairs (the better half of a bitonic merge), the 8 warp lists meet in
// shared memory behind one barrier and every thread merges them itself.  So
// every thread holds the support, sorted: its softmax, the integer ladder in
// index order and the next draft are computed by each thread from registers,
// and the Markov row of that draft is loaded without a further barrier.
constexpr int MK_THREADS = 256, MK_WARPS = MK_THREADS / 32;

__device__ __forceinline__ bool mk_better(float av, int ai, float bv, int bi) {
  return av > bv || (av == bv && ai < bi);
}

// v/ix (sorted, best first) <- the best KM of v/ix and ov/oi (both sorted)
template <int KM>
__device__ __forceinline__ void mk_merge(float (&v)[KM], int (&ix)[KM], const float (&ov)[KM], const int (&oi)[KM]) {
#pragma unroll
  for (int r = 0; r < KM; ++r)
    if (mk_better(ov[KM - 1 - r], oi[KM - 1 - r], v[r], ix[r])) {
      v[r] = ov[KM - 1 - r];
      ix[r] = oi[KM - 1 - r];
    }
  // v is now bitonic (worse towards the middle): half-cleaners sort it
#pragma unroll
  for (int h = KM / 2; h > 0; h >>= 1)
#pragma unroll
    for (int r = 0; r < KM; ++r)
      if ((r & h) == 0 && mk_better(v[r + h], ix[r + h], v[r], ix[r])) {
        const float tv = v[r];
        const int ti = ix[r];
        v[r] = v[r + h];
        ix[r] = ix[r + h];
        v[r + h] = tv;
        ix[r + h] = ti;
      }
}

template <int KM, int EM>
__global__ void __launch_bounds__(MK_THREADS) markov_draft_topk_kernel(
    const float* __restrict__ trunk, const float* __restrict__ M, int V, const int32_t* prev_dev,
    const float* __restrict__ u, int gamma, float T, int k, int mode, int32_t* drafts, float* q) {
  __shared__ float lv[2][MK_WARPS][KM];
  __shared__ int li[2][MK_WARPS][KM];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr int NONE = 0x7fffffff;
  pdl_trigger();
  pdl_wait();
  int prev = prev_dev[0];
  if (prev < 0 || prev >= V) prev = 0;
  float tr[EM];
#pragma unroll
  for (int e = 0; e < EM; ++e) {
    const int j = tid + MK_THREADS * e;
    tr[e] = (j < V && gamma > 0) ? trunk[j] : 0.f;
  }
  for (int i = 0; i < gamma; ++i) {
    const float* mr = M + (size_t)prev * V;
    const float* tn = trunk + (size_t)(i + 1) * V;
    float l[EM], tnx[EM];
#pragma unroll
    for (int e = 0; e < EM; ++e) {
      const int j = tid + MK_THREADS * e;
      l[e] = j < V ? __fadd_rn(tr[e], mr[j]) : 0.f;
      tnx[e] = (j < V && i + 1 < gamma) ? tn[j] : 0.f;
    }
    float v[KM];
    int ix[KM];
#pragma unroll
    for (int r = 0; r < KM; ++r) {
      v[r] = -INFINITY;
      ix[r] = NONE;
    }
#pragma unroll
    for (int e = 0; e < EM; ++e) {
      float x = l[e];
      int j = tid + MK_THREADS * e;
      if (j < V && mk_better(x, j, v[KM - 1], ix[KM - 1])) {
#pragma unroll
        for (int r = 0; r < KM; ++r)
          if (mk_better(x, j, v[r], ix[r])) {
            const float tv = v[r];
            const int ti = ix[r];
            v[r] = x;
            ix[r] = j;
            x = tv;
            j = ti;
          }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      float ov[KM];
      int oi[KM];
#pragma unroll
      for (int r = 0; r < KM; ++r) {
        ov[r] = __shfl_xor_sync(0xffffffffu, v[r], o);
        oi[r] = __shfl_xor_sync(0xffffffffu, ix[r], o);
      }
      mk_merge<KM>(v, ix, ov, oi);
    }
    const int b = i & 1;  // the barrier of slot i-1 ended every read of buffer b from slot i-2
    if (lane < KM) {
#pragma unroll
      for (int r = 0; r < KM; ++r)
        if (r == lane) {
          lv[b][warp][r] = v[r];
          li[b][warp][r] = ix[r];
        }
    }
    __syncthreads();
#pragma unroll
    for (int w = 0; w < MK_WARPS; ++w) {
      if (w == warp) continue;
      float ov[KM];
      int oi[KM];
#pragma unroll
      for (int r = 0; r < KM; ++r) {
        ov[r] = lv[b][w][r];
        oi[r] = li[b][w][r];
      }
      mk_merge<KM>(v, ix, ov, oi);
    }
    // the support: the first k entries; softmax of (l - max) / T over it
    const float mx = v[0];
    float w[KM], sum = 0.f;
#pragma unroll
    for (int r = 0; r < KM; ++r) {
      w[r] = (r < k && ix[r] != NONE) ? expf((v[r] - mx) / T) : 0.f;
      sum += w[r];
    }
#pragma unroll
    for (int r = 0; r < KM; ++r) w[r] = w[r] / sum;
    int d = -1;
    if (mode == EVS_SAMPLE) {
      unsigned int W[KM];
      unsigned long long S = 0;
#pragma unroll
      for (int r = 0; r < KM; ++r) {
        W[r] = ladder_weight(w[r]);
        S += W[r];
      }
      const unsigned long long U = min((unsigned long long)(unsigned int)(u[i] * 16777216.0f), 16777215ull);
      const unsigned long long thr = (U * S) >> 24;
      // the ladder in index order: entry r holds [pre_r, pre_r + W_r)
#pragma unroll
      for (int r = 0; r < KM; ++r) {
        unsigned long long pre = 0;
#pragma unroll
        for (int s2 = 0; s2 < KM; ++s2)
          if (ix[s2] < ix[r]) pre += W[s2];
        if (W[r] > 0 && pre <= thr && thr < pre + W[r]) d = ix[r];
      }
    }
    if (d < 0) d = ix[0] == NONE ? 0 : ix[0];  // greedy, or no integer mass: the argmax
#pragma unroll
    for (int e = 0; e < EM; ++e) {
      const int j = tid + MK_THREADS * e;
      if (j < V) {
        float qv = 0.f;
#pragma unroll
        for (int r = 0; r < KM; ++r)
          if (ix[r] == j) qv = w[r];
        q[(size_t)i * V + j] = qv;
      }
    }
    if (tid == 0) drafts[i] = d;
    prev = d;
#pragma unroll
    for (int e = 0; e < EM; ++e) tr[e] = tnx[e];
  }
}

// The top_k <= 8 chain by one warp when V <= 1024 and V % 4 == 0 (rows of
// whole float4s): lane l owns the NPL contiguous entries from l * NPL.  An
// entry's order is its orderable 32-bit key (NaN: key 0, never taken), ties
// to the lower index; a support round is one warp max of the lanes' best
// keys, a ballot for the lowest lane holding it (lowest lane = lowest
// index), and a rescan by that lane alone.  The support then sits in every
// lane's registers, and so do its softmax, the ladder draw and the next
// draft: the next Markov row is requested before this slot's q is stored
// (greedy: right after the first round, the draft being the argmax).
__device__ __forceinline__ float mk_val(unsigned int key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

template <int NPL>
__device__ __forceinline__ void mk_load_row(float (&x)[NPL], const float* __restrict__ row, int j0, int V) {
#pragma unroll
  for (int c = 0; c < NPL / 4; ++c) {
    float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
    if (j0 + 4 * c < V) f = *reinterpret_cast<const float4*>(row + j0 + 4 * c);
    x[4 * c] = f.x;
    x[4 * c + 1] = f.y;
    x[4 * c + 2] = f.z;
    x[4 * c + 3] = f.w;
  }
}

// this lane's best key and the lowest entry holding it (key 0: none)
template <int NPL>
__device__ __forceinline__ void mk_lane_best(const unsigned int (&key)[NPL], unsigned int& bk, int& be) {
  unsigned int t[NPL];
#pragma unroll
  for (int e = 0; e < NPL; ++e) t[e] = key[e];
#pragma unroll
  for (int h = NPL / 2; h > 0; h >>= 1)
#pragma unroll
    for (int e = 0; e < h; ++e) t[e] = max(t[e], t[e + h]);
  bk = t[0];
  unsigned int m = 0;
#pragma unroll
  for (int e = 0; e < NPL; ++e) m |= (key[e] == bk ? 1u : 0u) << e;
  be = __ffs(m) - 1;
}

template <int KM, int NPL>
__global__ void __launch_bounds__(32) markov_draft_warp_kernel(
    const float* __restrict__ trunk, const float* __restrict__ M, int V, const int32_t* prev_dev,
    const float* __restrict__ u, int gamma, float T, int k, int mode, int32_t* drafts, float* q) {
  constexpr int NONE = 0x7fffffff;
  const int lane = threadIdx.x, j0 = lane * NPL;
  const int nown = max(0, min(NPL, V - j0));
  pdl_trigger();
  pdl_wait();
  int prev = prev_dev[0];
  if (prev < 0 || prev >= V) prev = 0;
  float tr[NPL], x[NPL];
  if (gamma > 0) {
    mk_load_row<NPL>(tr, trunk, j0, V);
    mk_load_row<NPL>(x, M + (size_t)prev * V, j0, V);
  }
  for (int i = 0; i < gamma; ++i) {
    const bool more = i + 1 < gamma;
    float tn[NPL];
    if (more) mk_load_row<NPL>(tn, trunk + (size_t)(i + 1) * V, j0, V);
    const float ui = u[i];
    unsigned int key[NPL];
#pragma unroll
    for (int e = 0; e < NPL; ++e) key[e] = e < nown ? ord_key(__fadd_rn(tr[e], x[e])) : 0u;
    unsigned int bk;
    int be;
    // the lane's best and second-best entries (key 0: none); a lane whose
    // best is taken promotes its second and rescans only when it wins again
    mk_lane_best<NPL>(key, bk, be);
    unsigned int bk2;
    int be2;
    {
      unsigned int rest[NPL];
#pragma unroll
      for (int e = 0; e < NPL; ++e) rest[e] = e == be ? 0u : key[e];
      mk_lane_best<NPL>(rest, bk2, be2);
    }
    bool have2 = true;
    unsigned int taken = 0;  // bit e: entry e is in the support
    unsigned int sk[KM];
    int si[KM];
    int d = -1;
#pragma unroll
    for (int r = 0; r < KM; ++r) {
      sk[r] = 0u;
      si[r] = NONE;
      if (r < k) {
        const unsigned int mk = __reduce_max_sync(0xffffffffu, bk);
        if (mk != 0u) {
          const int wl = __ffs(__ballot_sync(0xffffffffu, bk == mk)) - 1;
          sk[r] = mk;
          si[r] = wl * NPL + __shfl_sync(0xffffffffu, be, wl);
          if (r + 1 < k && lane == wl) {
            taken |= 1u << be;
            if (have2) {
              bk = bk2;
              be = be2;
              have2 = false;
            } else {
              unsigned int rest[NPL];
#pragma unroll
              for (int e = 0; e < NPL; ++e) rest[e] = (taken >> e) & 1u ? 0u : key[e];
              mk_lane_best<NPL>(rest, bk, be);
            }
          }
        }
      }
      if (r == 0 && mode != EVS_SAMPLE) {
        d = si[0] == NONE ? 0 : si[0];
        if (more) mk_load_row<NPL>(x, M + (size_t)d * V, j0, V);
      }
    }
    float w[KM], sum = 0.f;
    const float mx = mk_val(sk[0]);
#pragma unroll
    for (int r = 0; r < KM; ++r) {
      w[r] = sk[r] != 0u ? expf((mk_val(sk[r]) - mx) / T) : 0.f;
      sum += w[r];
    }
#pragma unroll
    for (int r = 0; r < KM; ++r) w[r] = w[r] / sum;
    if (mode == EVS_SAMPLE) {
      unsigned int W[KM];
      unsigned long long S = 0;
#pragma unroll
      for (int r = 0; r < KM; ++r) {
        W[r] = ladder_weight(w[r]);
        S += W[r];
      }
      const unsigned long long U = min((unsigned long long)(unsigned int)(ui * 16777216.0f), 16777215ull);
      const unsigned long long thr = (U * S) >> 24;
#pragma unroll
      for (int r = 0; r < KM; ++r) {
        unsigned long long pre = 0;
#pragma unroll
        for (int s2 = 0; s2 < KM; ++s2)
          if (si[s2] < si[r]) pre += W[s2];
        if (W[r] > 0 && pre <= thr && thr < pre + W[r]) d = si[r];
      }
      if (d < 0) d = si[0] == NONE ? 0 : si[0];  // no integer mass: the argmax
      if (more) mk_load_row<NPL>(x, M + (size_t)d * V, j0, V);
    }
    // q: this lane's entries zero, then its support entries (same thread,
    // so the later store wins)
    float* qr = q + (size_t)i * V;
#pragma unroll
    for (int c = 0; c < NPL / 4; ++c)
      if (j0 + 4 * c < V) *reinterpret_cast<float4*>(qr + j0 + 4 * c) = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int r = 0; r < KM; ++r)
      if (si[r] != NONE && (unsigned int)(si[r] - j0) < (unsigned int)NPL) qr[si[r]] = w[r];
    if (lane == 0) drafts[i] = d;
    if (more) {
#pragma unroll
      for (int e = 0; e < NPL; ++e) tr[e] = tn[e];
    }
  }
}

template <int KM, int NPL>
static cudaError_t launch_markov_warp(const LaunchCtx& L, const float* trunk, const float* M, int V,
                                      const int32_t* prev, const float* u, int gamma, float T, int k, int mode,
                                      int32_t* drafts, float* q) {
  return launch(L, markov_draft_warp_kernel<KM, NPL>, dim3(1), dim3(32), 0, trunk, M, V, prev, u, gamma, T, k, mode,
                drafts, q);
}

template <int KM>
static cudaError_t launch_markov_topk(const LaunchCtx& L, const float* trunk, const float* M, int V, const int32_t* prev,
                                      const float* u, int gamma, float T, int k, int mode, int32_t* drafts, float* q) {
  const bool al16 = ((reinterpret_cast<uintptr_t>(trunk) | reinterpret_cast<uintptr_t>(M) |
                      reinterpret_cast<uintptr_t>(q)) & 15) == 0;
  if (V % 4 == 0 && al16) {
    if (V <= 128) return launch_markov_warp<KM, 4>(L, trunk, M, V, prev, u, gamma, T, k, mode, drafts, q);
    if (V <= 512) return launch_markov_warp<KM, 16>(L, trunk, M, V, prev, u, gamma, T, k, mode, drafts, q);
    if (V <= 1024) return launch_markov_warp<KM, 32>(L, trunk, M, V, prev, u, gamma, T, k, mode, drafts, q);
  }
  if (V <= 2 * MK_THREADS)
    return launch(L, markov_draft_topk_kernel<KM, 2>, dim3(1), dim3(MK_THREADS), 0, trunk, M, V, prev, u, gamma, T,
                  k, mode, drafts, q);
  if (V <= 8 * MK_THREADS)
    return launch(L, markov_draft_topk_kernel<KM, 8>, dim3(1), dim3(MK_THREADS), 0, trunk, M, V, prev, u, gamma, T,
                  k, mode, drafts, q);
  return launch(L, markov_draft_topk_kernel<KM, 32>, dim3(1), dim3(MK_THREADS), 0, trunk, M, V, prev, u, gamma, T, k,
                mode, drafts, q);
}

// Commit: keep = *acc_dev + 1 when acc_dev is given, else keep_host.
// n_explicit > 0 replaces book->pending_n (bare-book operator use).
__global__ void commit_kernel(evs_book* book, int keep_host, const int32_t* acc_dev, int n_explicit) {
  pdl_trigger();
  pdl_wait();
  if (threadIdx.x != 0) return;
  commit_one(book, acc_dev ? acc_dev[0] + 1 : keep_host, n_explicit);
}

// Fixed amount of arithmetic (no memory, no waits) that occupies the stream
// for a few milliseconds; ends after `iters` iterations whatever happens.
__global__ void busy_kernel(long long iters, float* sink) {
  float x = threadIdx.x;
  for (long long i = 0; i < iters; ++i) x = fmaf(x, 0.999999f, 1e-7f);
  if (x == -1.f) sink[0] = x;  // never true; keeps the loop
}

__global__ void book_set_kernel(evs_book* book, evs_book v) {
  pdl_trigger();
  pdl_wait();
  if (threadIdx.x == 0) *book = v;
}

}  // namespace

cudaError_t launch_embed_norm(const LaunchCtx& L, int dtype, const void* E, const int32_t* tokens,
                              const SeqRows& sr, int d, int V, float eps, float* X, void* xn,
                              const SeqPtrs<evs_book*>& book) {
  const int cl = row_cluster(d);
  const int n = sr.row0[sr.nseq];
  if (dtype == EVS_BF16)
    return launch_cl(L, cl, embed_norm_kernel<bf16>, dim3(cl, n), dim3(256), 0, (const bf16*)E, tokens, V, X, d,
                     eps, (bf16*)xn, sr, book);
  return launch_cl(L, cl, embed_norm_kernel<float>, dim3(cl, n), dim3(256), 0, (const float*)E, tokens, V, X, d,
                   eps, (float*)xn, sr, book);
}

bool resid_norm_ok(int d) { return resid_cluster(d) > 0; }

cudaError_t launch_resid_norm(const LaunchCtx& L, int dtype, float* X, const MixSrc& slots, int n, int d, float eps,
                              void* xn) {
  const int cl = resid_cluster(d);
  if (dtype != EVS_BF16 || !slots.ws || cl < 1) return cudaErrorInvalidValue;
  const int warps = d / TILE_M / cl;
  return launch_cl(L, cl, resid_norm_kernel<bf16>, dim3(cl, n), dim3(32 * warps), 0, X,
                   SrcSlots{slots.ws, slots.tab, slots.slot_rows}, d, eps, (bf16*)xn);
}

cudaError_t launch_norm_apply(const LaunchCtx& L, int dtype, const float* X, const float* ss, int n, int d,
                              float eps, void* xn) {
  const int ntiles = (d + TILE_M - 1) / TILE_M;
  const dim3 g((d + 255) / 256, n);
  if (dtype == EVS_BF16)
    return launch(L, norm_apply_kernel<bf16>, g, dim3(256), 0, X, ss, ntiles, d, eps, (bf16*)xn);
  return launch(L, norm_apply_kernel<float>, g, dim3(256), 0, X, ss, ntiles, d, eps, (float*)xn);
}

cudaError_t launch_mlp_act(const LaunchCtx& L, int dtype, const MixSrc& gu, int n, int F, bool il, void* h) {
  const dim3 g((F + 255) / 256, n);
  if (gu.ws) {
    if (dtype != EVS_BF16) return cudaErrorInvalidValue;
    return launch(L, mlp_act_kernel<bf16, SrcSlots>, g, dim3(256), 0, SrcSlots{gu.ws, gu.tab, gu.slot_rows}, F,
                  (int)il, (bf16*)h);
  }
  const SrcPlain<float> sf{(const float*)gu.p, 2 * F};
  if (dtype == EVS_BF16) return launch(L, mlp_act_kernel<bf16, SrcPlain<float>>, g, dim3(256), 0, sf, F, (int)il, (bf16*)h);
  return launch(L, mlp_act_kernel<float, SrcPlain<float>>, g, dim3(256), 0, sf, F, (int)il, (float*)h);
}

cudaError_t launch_probs(const LaunchCtx& L, const float* logits, int n, int V, float T, int top_k, float* p) {
  const size_t smem = sizeof(float) * 2 * V;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(probs_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  return launch(L, probs_kernel, dim3(n), dim3(256), smem, logits, V, T, top_k, p);
}

cudaError_t launch_accept(const LaunchCtx& L, const float* p, const float* q, const int32_t* drafts,
                          const float* u, int n, int V, int mode, int32_t* acc, int32_t* tok, evs_book* book,
                          bool commit) {
  return launch_accept_batch(L, p, q, drafts, u, one_seq(n), V, mode, acc, tok, one_ptr(book), commit);
}

cudaError_t launch_accept_batch(const LaunchCtx& L, const float* p, const float* q, const int32_t* drafts,
                                const float* u, const SeqRows& sr, int V, int mode, int32_t* acc, int32_t* tok,
                                const SeqPtrs<evs_book*>& books, bool commit) {
  int nmax = 0;
  for (int b = 0; b < sr.nseq; ++b) nmax = std::max(nmax, sr.row0[b + 1] - sr.row0[b]);
  const size_t smem = sizeof(unsigned int) * V + 2 * sizeof(int) * nmax;
  if (smem > 48 * 1024) {
    if (smem > 227 * 1024) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(accept_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  return launch(L, accept_kernel, dim3(sr.nseq), dim3(256), smem, p, q, drafts, u, sr, V, mode, acc, tok, books,
                (int)commit);
}

cudaError_t launch_markov_draft(const LaunchCtx& L, const float* trunk, const float* M, int V, const int32_t* prev,
                                const float* u, int gamma, float T, int top_k, int mode, int32_t* drafts, float* q) {
  if (top_k > 0 && top_k < V && top_k <= 8 && V <= 32 * MK_THREADS) {
    if (top_k <= 4) return launch_markov_topk<4>(L, trunk, M, V, prev, u, gamma, T, top_k, mode, drafts, q);
    return launch_markov_topk<8>(L, trunk, M, V, prev, u, gamma, T, top_k, mode, drafts, q);
  }
  const size_t smem = sizeof(float) * 3 * V;
  if (smem > 48 * 1024) {
    if (smem > 200 * 1024) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(markov_draft_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  return launch(L, markov_draft_kernel, dim3(1), dim3(256), smem, trunk, M, V, prev, u, gamma, T, top_k, mode, drafts,
                q);
}

cudaError_t launch_commit(const LaunchCtx& L, evs_book* book, int keep, const int32_t* acc_dev, int n_explicit) {
  return launch(L, commit_kernel, dim3(1), dim3(32), 0, book, keep, acc_dev, n_explicit);
}

cudaError_t launch_book_set(const LaunchCtx& L, evs_book* book, evs_book v) {
  return launch(L, book_set_kernel, dim3(1), dim3(32), 0, book, v);
}

cudaError_t launch_busy(const LaunchCtx& L, long long iters) {
  return launch(L, busy_kernel, dim3(1), dim3(32), 0, iters, (float*)nullptr);
}

}  // namespace evs
