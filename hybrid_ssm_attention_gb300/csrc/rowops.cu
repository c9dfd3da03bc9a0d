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
// A cluster of CL CTAs per row, CTA = G groups of 128 threads; thread j of
// group g owns column j of each of the group's TPC consecutive 128-column
// tiles, so the sums of squares follow the GEMM_RESID epilogue exactly: per
// tile, x^2 of each warp's 32 columns by xor butterfly (16, 8, 4, 2, 1),
// then the four warps in order; the row's sum is the tile sums in tile
// order.  Each CTA pushes its tile sums into every CTA's shared memory
// before the one cluster barrier, after which only local memory is read.
template <typename T, int TPC>
__global__ void __launch_bounds__(256) resid_norm_kernel(float* X, const __grid_constant__ SrcSlots src, int d,
                                                         float eps, T* xn) {
  __shared__ float s_red[2][4][TPC];
  __shared__ float s_all[RESID_TILES_ROW];  // the row's tile sums, tile order
  __shared__ float s_den, s_rcp;
  cg::cluster_group cl = cg::this_cluster();
  const int ncl = (int)cl.num_blocks(), rank = (int)cl.block_rank();
  const int G = blockDim.x / TILE_M;
  const int t = blockIdx.y, g = threadIdx.x / TILE_M, j = threadIdx.x % TILE_M;
  const int ntiles = d / TILE_M, kc = rank * G * TPC, k0 = kc + g * TPC;
  const int lane = j & 31, w = j >> 5;
  pdl_trigger();
  SrcSlots::Col cs[TPC];
#pragma unroll
  for (int i = 0; i < TPC; ++i) cs[i] = src.at((k0 + i) * TILE_M + j);
  pdl_wait();
  float* xr = X + (size_t)t * d + j;
  // every load before the first store (X may alias the slots for all the
  // compiler knows); a tile has up to six stream-K contributors here
  float x[TPC], sv[TPC];
#pragma unroll
  for (int i = 0; i < TPC; ++i) {
    x[i] = __ldcg(xr + (k0 + i) * TILE_M);
    sv[i] = src.get<6>(cs[i], t, (k0 + i) * TILE_M + j);
  }
#pragma unroll
  for (int i = 0; i < TPC; ++i) {
    x[i] += sv[i];
    xr[(k0 + i) * TILE_M] = x[i];
    float sq = x[i] * x[i];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
    if (lane == 0) s_red[g][w][i] = sq;
  }
  __syncthreads();
  // tile sum (g, i) -> position kc + g*TPC + i of every CTA's s_all
  if (threadIdx.x < ncl * G * TPC) {
    const int q = threadIdx.x / (G * TPC), e = threadIdx.x % (G * TPC), gg = e / TPC, i = e % TPC;
    const float v = ((s_red[gg][0][i] + s_red[gg][1][i]) + s_red[gg][2][i]) + s_red[gg][3][i];
    *cl.map_shared_rank(&s_all[kc + e], q) = v;
  }
  cl.sync();
  if (threadIdx.x < 32) {
    // the tile sums, 32 at a time, added in tile order
    float tot = 0.f;
    for (int q0 = 0; q0 < ntiles; q0 += 32) {
      const float mine = q0 + lane < ntiles ? s_all[q0 + lane] : 0.f;
      for (int q = 0; q < 32 && q0 + q < ntiles; ++q) tot += __shfl_sync(0xffffffffu, mine, q);
    }
    if (lane == 0) {
      s_den = sqrtf(tot / (float)d + eps);
      s_rcp = 1.f / s_den;
    }
  }
  __syncthreads();
  T* xo = xn + (size_t)t * d + j;
#pragma unroll
  for (int i = 0; i < TPC; ++i) xo[(k0 + i) * TILE_M] = from_f<T>(div_row(x[i], s_den, s_rcp));
}

// Shape of the row split: G groups of 128 threads (2 if the tile count is
// even), CL CTAs (the largest of 4, 2, 1 that leaves a power-of-two TPC <=
// RESID_TILES_MAX tiles per group).  False if none fits.
bool resid_shape(int d, int* G, int* TPC, int* CL) {
  if (d % TILE_M || d / TILE_M > RESID_TILES_ROW) return false;
  const int nt = d / TILE_M;
  *G = nt % 2 == 0 ? 2 : 1;
  const int rest = nt / *G;
  for (int cl = 4; cl >= 1; cl >>= 1) {
    const int tpc = rest / cl;
    if (rest % cl == 0 && tpc <= RESID_TILES_MAX && (tpc & (tpc - 1)) == 0) {
      *TPC = tpc;
      *CL = cl;
      return true;
    }
  }
  return false;
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

// One CTA per row.  top-k by rank: entry j is kept iff fewer than k entries
// beat it (larger value, or equal value at a lower index).
__global__ void __launch_bounds__(256) probs_kernel(const float* logits, int V, float T, int k, float* p) {
  extern __shared__ float sm[];
  __shared__ float scratch[32];
  float* l_s = sm;        // [V]
  float* w_s = sm + V;    // [V]
  const int t = blockIdx.x;
  pdl_trigger();
  pdl_wait();
  for (int j = threadIdx.x; j < V; j += blockDim.x) l_s[j] = logits[(size_t)t * V + j];
  __syncthreads();
  const bool use_k = k > 0 && k < V;
  float mx = -INFINITY;
  for (int j = threadIdx.x; j < V; j += blockDim.x) {
    bool keep = true;
    if (use_k) {
      const float lj = l_s[j];
      int rank = 0;
      for (int l = 0; l < V; ++l) rank += (l_s[l] > lj) || (l_s[l] == lj && l < j);
      keep = rank < k;
    }
    w_s[j] = keep ? 1.f : 0.f;
    if (keep) mx = fmaxf(mx, l_s[j]);
  }
  mx = block_reduce(mx, MaxF(), scratch);
  float sum = 0.f;
  for (int j = threadIdx.x; j < V; j += blockDim.x) {
    const float w = w_s[j] != 0.f ? expf((l_s[j] - mx) / T) : 0.f;
    w_s[j] = w;
    sum += w;
  }
  sum = block_reduce(sum, AddF(), scratch);
  for (int j = threadIdx.x; j < V; j += blockDim.x) p[(size_t)t * V + j] = w_s[j] / sum;
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

__global__ void __launch_bounds__(256) accept_kernel(const float* p, const float* q, const int32_t* drafts,
                                                     const float* u, int n, int V, int mode, int32_t* out_a,
                                                     int32_t* out_tok) {
  extern __shared__ unsigned int Wsm[];  // [V], then s_arg[n], s_ok[n]
  __shared__ unsigned long long us[256];
  __shared__ int found;
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
    const unsigned long long U = (unsigned long long)(unsigned int)(u[gamma] * 16777216.0f);
    const unsigned long long thr = (U * S) >> 24;
    token = ladder_find(Wsm, V, thr, us, &found);
  }
  if (threadIdx.x == 0) {
    out_a[0] = a;
    out_tok[0] = token;
  }
}

// Commit: keep = *acc_dev + 1 when acc_dev is given, else keep_host.
// n_explicit > 0 replaces book->pending_n (bare-book operator use).
__global__ void commit_kernel(evs_book* book, int keep_host, const int32_t* acc_dev, int n_explicit) {
  pdl_trigger();
  pdl_wait();
  if (threadIdx.x != 0) return;
  const int keep = acc_dev ? acc_dev[0] + 1 : keep_host;
  const int n = n_explicit > 0 ? n_explicit : book->pending_n;
  if (n <= 0 || keep < 0 || keep > n) {
    set_status(book, EVS_DEV_BAD_KEEP);
    book->pending_n = 0;
    return;
  }
  book->fir_bank ^= 1;
  book->fir_off = keep;
  if (keep > 0) {
    book->iir_bank ^= 1;
    book->iir_slot = keep - 1;
  }
  book->pos += keep;
  book->pending_n = 0;
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

bool resid_norm_ok(int d) {
  int G, TPC, CL;
  return resid_shape(d, &G, &TPC, &CL);
}

cudaError_t launch_resid_norm(const LaunchCtx& L, int dtype, float* X, const MixSrc& slots, int n, int d, float eps,
                              void* xn) {
  int G, TPC, CL;
  if (dtype != EVS_BF16 || !slots.ws || !resid_shape(d, &G, &TPC, &CL)) return cudaErrorInvalidValue;
  const SrcSlots src{slots.ws, slots.tab, slots.slot_rows};
  void (*k)(float*, SrcSlots, int, float, bf16*);
  switch (TPC) {
    case 1: k = resid_norm_kernel<bf16, 1>; break;
    case 2: k = resid_norm_kernel<bf16, 2>; break;
    case 4: k = resid_norm_kernel<bf16, 4>; break;
    case 8: k = resid_norm_kernel<bf16, 8>; break;
    case 16: k = resid_norm_kernel<bf16, 16>; break;
    default: return cudaErrorInvalidValue;
  }
  return launch_cl(L, CL, k, dim3(CL, n), dim3(G * TILE_M), 0, X, src, d, eps, (bf16*)xn);
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
                          const float* u, int n, int V, int mode, int32_t* acc, int32_t* tok) {
  const size_t smem = sizeof(unsigned int) * V + 2 * sizeof(int) * n;
  if (smem > 48 * 1024) {
    if (smem > 227 * 1024) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(accept_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  return launch(L, accept_kernel, dim3(1), dim3(256), smem, p, q, drafts, u, n, V, mode, acc, tok);
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
