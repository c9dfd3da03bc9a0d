// Sequence mixers of the hybrid stack for one verify block, each keeping the
// state after every block position ("What we implemented" in the EvSpark
// discussion post; author's reply, prerequisite 1):
//
//  FIR  (short / medium Hyena filter): the inputs live in a ring of
//       R = L-1+n_max rows, position p at row p mod R.  The committed window
//       is positions pos-L+1 .. pos-1; the kernel writes the block's inputs
//       at positions pos .. pos+n-1, so every block position's window is in
//       place and commit only moves pos (no copy).
//  IIR  (modal Hyena filter): s_t = lam * s_{t-1} + z_t per channel and pole,
//       y_t = Re sum_m R_m s_t[m]; all n states go to the spare bank.
//  ATTN rotary q/k, append k/v at rows pos..pos+n-1 (append-only cache),
//       split-KV block-causal attention with a fixed-order combine.  Here:
//       the SIMT path for float caches and head dims without tensor maps;
//       bf16 caches at Dh 64 / 128 take the tensor-map kernel (attention.cu)
//       and share the combine.
//
// Every mixer first forms its inputs from the in-projection (GEMM partials
// or a plain matrix) with the storage rounding of the path.
#include <algorithm>
#include <cmath>

#include "evs_internal.cuh"

namespace evs {
namespace {

// 16-byte global -> shared copy that does not block the issuing thread;
// cp_async_wait_all() waits for all of the thread's outstanding copies.
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(smem_dst)),
               "l"(gmem_src)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// ------------------------------------------------------------------ FIR
// Block = 32 channels x NW warps; warp w sums taps [w*J, (w+1)*J), J = JT.
// Each lane keeps its J taps and the J + 15 window values they touch in
// registers.  Shared rows: the window (positions pos-L+1 .. pos-1) followed
// by the block's inputs.
template <typename T, typename Src, int JT>
__global__ void __launch_bounds__(256)
    fir_kernel(Src src, int d, int Lf, int R, const float* __restrict__ taps, const __grid_constant__ SeqRows sr,
               const __grid_constant__ SeqPtrs<float*> rings, const __grid_constant__ SeqPtrs<const evs_book*> books,
               T* g) {
  extern __shared__ float sm[];
  const int NW = blockDim.x >> 5;
  // this CTA's sequence: block rows [r0, r0 + n), its own ring and bookkeeping
  const int sq = blockIdx.y, r0 = sr.row0[sq], n = sr.row0[sq + 1] - r0;
  float* ring = rings.p[sq];
  const evs_book* book = books.p[sq];
  const int rows = Lf - 1 + n;
  float* ext_s = sm;                       // [rows][32]
  float* a_s = ext_s + rows * 32;          // [n][32]
  float* tap_s = a_s + n * 32;             // [Lf][32]
  float* part_s = tap_s + Lf * 32;         // [NW][n][32]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c0 = blockIdx.x * 32, c = c0 + lane;

  pdl_trigger();
  // Taps and the committed window do not depend on the in-projection: loaded
  // while the preceding GEMM still runs (pos is fixed for the whole verify).
  const long long pos = book->pos;
  // rows of 32 channels = 128 bytes = 8 x 16-byte pieces, all copies in flight at once
  const int nthr = blockDim.x;
  for (int e = threadIdx.x; e < Lf * 8; e += nthr) {
    const int j = e >> 3, w = e & 7;
    cp_async16(tap_s + j * 32 + w * 4, taps + (size_t)j * d + c0 + w * 4);
  }
  for (int e = threadIdx.x; e < (Lf - 1) * 8; e += nthr) {
    const int r = e >> 3, w = e & 7;
    const long long p = pos - (Lf - 1) + r;  // >= -(Lf - 1) > -R: rows before position 0 hold zeros
    const int pr = (int)(p >= 0 ? p % R : p + R);
    cp_async16(ext_s + r * 32 + w * 4, ring + (size_t)pr * d + c0 + w * 4);
  }
  const auto ca = src.at(c), cb = src.at(d + c), cv = src.at(2 * d + c);
  cp_async_wait_all();
  __syncthreads();
  pdl_wait();
  // three of this warp's rows at a time, all reads issued before any use
  // (rows past the block re-read its last row and are dropped)
  for (int t0 = warp; t0 < n; t0 += 3 * NW) {
    float av[3], bv[3], vv[3];
#pragma unroll
    for (int k = 0; k < 3; ++k) {
      const int t = min(t0 + k * NW, n - 1);
      av[k] = src.get(ca, r0 + t, c);
      bv[k] = src.get(cb, r0 + t, d + c);
      vv[k] = src.get(cv, r0 + t, 2 * d + c);
    }
#pragma unroll
    for (int k = 0; k < 3; ++k) {
      const int t = t0 + k * NW;
      if (t < n) {
        const float a = stored<T>(av[k]), b = stored<T>(bv[k]), v = stored<T>(vv[k]);
        a_s[t * 32 + lane] = a;
        ext_s[(Lf - 1 + t) * 32 + lane] = b * v;
        ring[(size_t)((pos + t) % R) * d + c] = b * v;
      }
    }
  }
  __syncthreads();
  // y_t partial = sum_{j in [j0, j0+JT), j < Lf} h[j] * ext[Lf-1+t-j]; the
  // window rows used are base .. base+JT+NTOK-2 with base = Lf-1-j0-(JT-1)
  const int j0 = warp * JT;
  const int base = Lf - 1 - j0 - (JT - 1);
  float hreg[JT];
  float wreg[JT + NTOK - 1];
#pragma unroll
  for (int q = 0; q < JT; ++q) hreg[q] = (j0 + q < Lf) ? tap_s[(j0 + q) * 32 + lane] : 0.f;
#pragma unroll
  for (int q = 0; q < JT + NTOK - 1; ++q) {
    const int p = base + q;
    wreg[q] = (p >= 0 && p < rows) ? ext_s[p * 32 + lane] : 0.f;
  }
  // all NTOK rows in one block so the per-row FMA chains interleave (rows
  // past the block read zero window values and are not stored)
  float acc[NTOK];
#pragma unroll
  for (int t = 0; t < NTOK; ++t) {
    acc[t] = 0.f;
#pragma unroll
    for (int q = 0; q < JT; ++q)
      if (j0 + q < Lf) acc[t] = fmaf(hreg[q], wreg[t - q + JT - 1], acc[t]);
  }
#pragma unroll
  for (int t = 0; t < NTOK; ++t)
    if (t < n) part_s[(warp * n + t) * 32 + lane] = acc[t];
  __syncthreads();
  for (int t = warp; t < n; t += NW) {
    float y = 0.f;
    for (int w = 0; w < NW; ++w) y += part_s[(w * n + t) * 32 + lane];
    g[(size_t)(r0 + t) * d + c] = from_f<T>(a_s[t * 32 + lane] * y);
  }
}

// ------------------------------------------------------------------ IIR
// Block = 256 threads = (256/M) channels x M poles, poles of a channel in
// adjacent lanes.  Per-position states land in the spare bank [n][d][M].
template <typename T, typename Src, int M>
__global__ void __launch_bounds__(256)
    iir_kernel(Src src, int d, const float2* __restrict__ lam, const float2* __restrict__ res,
               const __grid_constant__ SeqRows sr, const __grid_constant__ SeqPtrs<float2*> st0s,
               const __grid_constant__ SeqPtrs<float2*> st1s, const __grid_constant__ SeqPtrs<const evs_book*> books,
               T* g) {
  constexpr int CPB = 256 / M;
  // this CTA's sequence: block rows [r0, r0 + n), its own banks and bookkeeping
  const int sq = blockIdx.y, r0 = sr.row0[sq], n = sr.row0[sq + 1] - r0;
  float2* st0 = st0s.p[sq];
  float2* st1 = st1s.p[sq];
  const evs_book* book = books.p[sq];
  __shared__ float z_s[NTOK][CPB];
  __shared__ float a_s[NTOK][CPB];
  const int cl = threadIdx.x / M, m = threadIdx.x % M;
  const int c = blockIdx.x * CPB + cl;
  pdl_trigger();
  // poles, residues and the committed state do not depend on the
  // in-projection: loaded while the preceding GEMM still runs
  const float2 L = lam[(size_t)c * M + m];
  const float2 R = res[(size_t)c * M + m];
  const int bank = book->iir_bank, slot = book->iir_slot;
  const float2* cur = bank ? st1 : st0;
  float2* dst = bank ? st0 : st1;
  float2 s = make_float2(0.f, 0.f);
  if (slot >= 0) s = cur[((size_t)slot * d + c) * M + m];
  // 256 is a multiple of CPB: this thread's staging column is fixed
  const int cc = blockIdx.x * CPB + threadIdx.x % CPB;
  const auto ca = src.at(cc), cb = src.at(d + cc), cv = src.at(2 * d + cc);
  pdl_wait();
  for (int e = threadIdx.x; e < n * CPB; e += 256) {
    const int t = e / CPB;
    const float a = stored<T>(src.get(ca, r0 + t, cc));
    const float b = stored<T>(src.get(cb, r0 + t, d + cc));
    const float v = stored<T>(src.get(cv, r0 + t, 2 * d + cc));
    a_s[t][e % CPB] = a;
    z_s[t][e % CPB] = b * v;
  }
  __syncthreads();
  for (int t = 0; t < n; ++t) {
    const float z = z_s[t][cl];
    const float sr = fmaf(L.x, s.x, fmaf(-L.y, s.y, z));
    const float si = fmaf(L.x, s.y, L.y * s.x);
    s = make_float2(sr, si);
    dst[((size_t)t * d + c) * M + m] = s;
    float y = fmaf(R.x, s.x, -R.y * s.y);
#pragma unroll
    for (int o = M / 2; o > 0; o >>= 1) y += __shfl_xor_sync(0xffffffffu, y, o);
    if (m == 0) g[(size_t)(r0 + t) * d + c] = from_f<T>(a_s[t][cl] * y);
  }
}

// ------------------------------------------------------------------ attention
// (1) rotary embedding + append: grid (n, H), Dh/2 threads, one rotation pair each.
template <typename T, typename Src>
__global__ void qkv_rope_kernel(Src src, int H, int Dh, long long ctx_max, const uint64_t* turn_fx,
                                const __grid_constant__ SeqRows sr, const __grid_constant__ SeqPtrs<T*> kcs,
                                const __grid_constant__ SeqPtrs<T*> vcs, float* qbuf,
                                const __grid_constant__ SeqPtrs<evs_book*> books) {
  // block row r: position t of sequence sq
  const int r = blockIdx.x, h = blockIdx.y, i = threadIdx.x, half = Dh >> 1;
  const int sq = seq_of_row(sr, r), t = r - sr.row0[sq];
  T* kc = kcs.p[sq];
  T* vc = vcs.p[sq];
  evs_book* book = books.p[sq];
  const int d = H * Dh;
  pdl_trigger();
  // the position is fixed for the whole verify: the rotation is computed
  // while the in-projection still runs
  const long long pos = (long long)book->pos + t;
  const float2 c = rope_cs(pos, turn_fx[i]);
  const int col = h * Dh + i;
  const auto cq1 = src.at(col), cq2 = src.at(col + half), ck1 = src.at(d + col), ck2 = src.at(d + col + half);
  const auto cv1 = src.at(2 * d + col), cv2 = src.at(2 * d + col + half);
  pdl_wait();
  if (pos >= ctx_max) {
    if (i == 0) set_status(book, EVS_DEV_KV_OVERFLOW);
    return;
  }
  const float q1 = stored<T>(src.get(cq1, r, col)), q2 = stored<T>(src.get(cq2, r, col + half));
  const float k1 = stored<T>(src.get(ck1, r, d + col)), k2 = stored<T>(src.get(ck2, r, d + col + half));
  const float v1 = stored<T>(src.get(cv1, r, 2 * d + col)), v2 = stored<T>(src.get(cv2, r, 2 * d + col + half));
  const float rq1 = rot_lo(q1, q2, c), rq2 = rot_hi(q1, q2, c);
  const float rk1 = rot_lo(k1, k2, c), rk2 = rot_hi(k1, k2, c);
  const size_t row = ((size_t)h * ctx_max + pos) * Dh;
  kc[row + i] = from_f<T>(rk1);
  kc[row + i + half] = from_f<T>(rk2);
  vc[row + i] = from_f<T>(v1);
  vc[row + i + half] = from_f<T>(v2);
  float* qo = qbuf + ((size_t)r * H + h) * Dh;
  qo[i] = stored<T>(rq1);
  qo[i + half] = stored<T>(rq2);
}

// (2) split-KV (SIMT, any storage type): CTA (s, h) owns the keys of split s,
// [s*span, (s+1)*span), and walks them in chunks of CH keys at absolute
// positions.  Query t (position pos+t) sees keys <= pos+t.  Each chunk's K
// and V rows are staged in shared memory (K rows padded by 16 bytes so the
// per-key dot products of a warp hit distinct banks); per chunk and query
// the kernel forms the max, the sum of exp and the unnormalised output and
// folds them into the split's running (max, sum, output).  Every reduction
// runs over fixed key slots, masked slots contributing exact zeros, so a
// query's result does not depend on the other queries of the block.
template <typename T, int DH, int CH>
__global__ void __launch_bounds__(256)
    attn_split_kernel(const float* __restrict__ qbuf, const __grid_constant__ SeqPtrs<const T*> kcs,
                      const __grid_constant__ SeqPtrs<const T*> vcs, int H, const __grid_constant__ SeqRows sr,
                      long long ctx_max, const __grid_constant__ SeqPtrs<const evs_book*> books, int span,
                      const __grid_constant__ SeqPtrs<float*> part_os, const __grid_constant__ SeqPtrs<float*> part_mls,
                      int nsplit_max) {
  constexpr int KP = DH * (int)sizeof(T) + 16;  // padded K row pitch in bytes
  constexpr int VP = DH * (int)sizeof(T);
  constexpr int QG = 256 / CH;                   // query groups in the score phase
  constexpr int QS = NTOK / QG > 0 ? NTOK / QG : 1;
  constexpr int DP = DH / 2;                     // output dim pairs
  constexpr int OG = 256 / DP;                   // query groups in the PV phase
  constexpr int OS = (NTOK + OG - 1) / OG;
  extern __shared__ __align__(16) unsigned char smraw[];
  float* q_s = reinterpret_cast<float*>(smraw);                    // [NTOK][DH]
  float* p_s = q_s + NTOK * DH;                                    // [NTOK][CH]
  float* ml_s = p_s + NTOK * CH;                                   // [NTOK][4]: running max, sum; chunk weights
  unsigned char* k_s = reinterpret_cast<unsigned char*>(ml_s + NTOK * 4);  // [CH][KP]
  unsigned char* v_s = k_s + CH * KP;                              // [CH][VP]
  const int h = blockIdx.y, sp = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // this CTA's sequence (blockIdx.z): its queries are block rows [r0, r0 + n)
  const int sq = blockIdx.z, r0 = sr.row0[sq], n = sr.row0[sq + 1] - r0;
  const T* kc = kcs.p[sq];
  const T* vc = vcs.p[sq];
  const evs_book* book = books.p[sq];
  float* part_o = part_os.p[sq];
  float* part_ml = part_mls.p[sq];
  pdl_trigger();
  // the committed length is fixed for the whole verify: pull this split's
  // committed keys / values into L2 while the in-projection still runs
  const long long pos = book->pos;
  const long long total = min(pos + n, ctx_max);
  const long long kb0 = (long long)sp * span, kb1 = min(kb0 + span, total);
  if (tid == 0) {
    const long long pre_end = min(kb1, min(pos, ctx_max));
    if (pre_end > kb0) {
      const unsigned bytes = (unsigned)((pre_end - kb0) * DH * sizeof(T));
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(kc + ((size_t)h * ctx_max + kb0) * DH),
                   "r"(bytes)
                   : "memory");
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(vc + ((size_t)h * ctx_max + kb0) * DH),
                   "r"(bytes)
                   : "memory");
    }
  }
  pdl_wait();
  if (kb0 >= total) return;  // this split holds no key of the block
  const float scale = rsqrtf((float)DH);
  for (int e = tid; e < NTOK * DH; e += 256) {
    const int t = e / DH;
    q_s[e] = t < n ? qbuf[((size_t)(r0 + t) * H + h) * DH + e % DH] : 0.f;
  }
  if (tid < NTOK) {
    ml_s[tid * 4] = -INFINITY;
    ml_s[tid * 4 + 1] = 0.f;
  }
  const int dp = tid % DP, tqo = tid / DP;
  float ra[OS], rb[OS];  // running unnormalised output
#pragma unroll
  for (int r = 0; r < OS; ++r) ra[r] = rb[r] = 0.f;
  for (long long k0 = kb0; k0 < kb1; k0 += CH) {
    const int kmax = (int)min((long long)CH, kb1 - k0);
    __syncthreads();
    // stage K and V rows [k0, k0+kmax) with 16-byte loads
    constexpr int VEC = DH * (int)sizeof(T) / 16;  // 16-byte vectors per row
    for (int e = tid; e < kmax * VEC; e += 256) {
      const int j = e / VEC, w = e % VEC;
      cp_async16(k_s + j * KP + w * 16, kc + ((size_t)h * ctx_max + k0 + j) * DH + w * 16 / sizeof(T));
      cp_async16(v_s + j * VP + w * 16, vc + ((size_t)h * ctx_max + k0 + j) * DH + w * 16 / sizeof(T));
    }
    cp_async_wait_all();
    __syncthreads();
    // scores: thread = (key slot j, query group tq)
    {
      const int j = tid % CH, tq = tid / CH;
      float dots[QS];
#pragma unroll
      for (int r = 0; r < QS; ++r) dots[r] = 0.f;
      if (j < kmax) {
#pragma unroll 4
        for (int w = 0; w < VEC; ++w) {
          const uint4 raw = *reinterpret_cast<const uint4*>(k_s + j * KP + w * 16);
          float kv[16 / sizeof(T)];
          if constexpr (sizeof(T) == 2) {
            const bf16* b = reinterpret_cast<const bf16*>(&raw);
#pragma unroll
            for (int z = 0; z < 8; ++z) kv[z] = __bfloat162float(b[z]);
          } else {
            const float* f = reinterpret_cast<const float*>(&raw);
#pragma unroll
            for (int z = 0; z < 4; ++z) kv[z] = f[z];
          }
          constexpr int EPV = 16 / sizeof(T);
#pragma unroll
          for (int r = 0; r < QS; ++r) {
            const int t = tq + r * QG;
            if (t < n) {
#pragma unroll
              for (int z = 0; z < EPV; ++z) dots[r] = fmaf(q_s[t * DH + w * EPV + z], kv[z], dots[r]);
            }
          }
        }
      }
#pragma unroll
      for (int r = 0; r < QS; ++r) {
        const int t = tq + r * QG;
        if (t < n) {
          const long long kp = k0 + j;
          p_s[t * CH + j] = (j < kmax && kp <= pos + t) ? dots[r] * scale : -INFINITY;
        }
      }
    }
    __syncthreads();
    // per query: the chunk's max and sum of exp, folded into the running pair
    // (warp per query; the weights of old and new go to ml_s[t][2..3])
    for (int t = warp; t < n; t += 8) {
      float mx = -INFINITY;
      for (int j = lane; j < CH; j += 32) mx = fmaxf(mx, p_s[t * CH + j]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      float sum = 0.f;
      for (int j = lane; j < CH; j += 32) {
        const float sc = p_s[t * CH + j];
        const float p = (mx == -INFINITY || sc == -INFINITY) ? 0.f : expf(sc - mx);
        p_s[t * CH + j] = p;
        sum += p;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      if (lane == 0) {
        const float M = ml_s[t * 4], Mn = fmaxf(M, mx);
        const float wo = Mn == -INFINITY ? 1.f : expf(M - Mn);
        const float wc = mx == -INFINITY ? 0.f : expf(mx - Mn);
        ml_s[t * 4] = Mn;
        ml_s[t * 4 + 1] = fmaf(ml_s[t * 4 + 1], wo, sum * wc);
        ml_s[t * 4 + 2] = wo;
        ml_s[t * 4 + 3] = wc;
      }
    }
    __syncthreads();
    // chunk output, folded into the running output: thread = (dim pair, query group)
    {
      float o0[OS], o1[OS];
#pragma unroll
      for (int r = 0; r < OS; ++r) o0[r] = o1[r] = 0.f;
#pragma unroll 4
      for (int j = 0; j < kmax; ++j) {
        float v0, v1;
        if constexpr (sizeof(T) == 2) {
          const __nv_bfloat162 vv = *reinterpret_cast<const __nv_bfloat162*>(v_s + j * VP + dp * 4);
          v0 = __low2float(vv);
          v1 = __high2float(vv);
        } else {
          const float2 vv = *reinterpret_cast<const float2*>(v_s + j * VP + dp * 8);
          v0 = vv.x;
          v1 = vv.y;
        }
#pragma unroll
        for (int r = 0; r < OS; ++r) {
          const int t = tqo + r * OG;
          if (t < n) {
            const float p = p_s[t * CH + j];
            o0[r] = fmaf(p, v0, o0[r]);
            o1[r] = fmaf(p, v1, o1[r]);
          }
        }
      }
#pragma unroll
      for (int r = 0; r < OS; ++r) {
        const int t = tqo + r * OG;
        if (t < n) {
          const float wo = ml_s[t * 4 + 2], wc = ml_s[t * 4 + 3];
          ra[r] = fmaf(ra[r], wo, o0[r] * wc);
          rb[r] = fmaf(rb[r], wo, o1[r] * wc);
        }
      }
    }
  }
#pragma unroll
  for (int r = 0; r < OS; ++r) {
    const int t = tqo + r * OG;
    if (t < n) {
      float* o = part_o + (((size_t)h * nsplit_max + sp) * NTOK + t) * DH + 2 * dp;
      o[0] = ra[r];
      o[1] = rb[r];
    }
  }
  if (tid < n) {
    float* ml = part_ml + (((size_t)h * nsplit_max + sp) * NTOK + tid) * 2;
    ml[0] = ml_s[tid * 4];
    ml[1] = ml_s[tid * 4 + 1];
  }
}

// (3) combine: grid (n, H), Dh threads; splits in ascending order.
template <typename T>
__global__ void attn_combine_kernel(const __grid_constant__ SeqPtrs<const float*> part_os,
                                    const __grid_constant__ SeqPtrs<const float*> part_mls, int H, int Dh,
                                    const __grid_constant__ SeqRows sr, int span, long long ctx_max,
                                    const __grid_constant__ SeqPtrs<const evs_book*> books,
                                    int nsplit_max, T* g) {
  // block row r: query t of sequence sq
  const int r = blockIdx.x, h = blockIdx.y, e = threadIdx.x;
  const int sq = seq_of_row(sr, r), t = r - sr.row0[sq];
  const float* part_o = part_os.p[sq];
  const float* part_ml = part_mls.p[sq];
  const evs_book* book = books.p[sq];
  pdl_trigger();
  pdl_wait();
  const long long qpos = min((long long)book->pos + t, ctx_max - 1);
  const int nc = (int)(qpos / span) + 1;  // splits holding keys <= qpos
  const float* ml = part_ml + ((size_t)h * nsplit_max * NTOK + t) * 2;
  float M = -INFINITY;
#pragma unroll 8
  for (int c = 0; c < nc; ++c) M = fmaxf(M, ml[(size_t)c * NTOK * 2]);
  float l = 0.f, o = 0.f;
  // loads are independent of the running sums: unrolled so they overlap
#pragma unroll 8
  for (int c = 0; c < nc; ++c) {
    const float mc = ml[(size_t)c * NTOK * 2];
    const float lc = ml[(size_t)c * NTOK * 2 + 1];
    const float oc = part_o[(((size_t)h * nsplit_max + c) * NTOK + t) * Dh + e];
    if (mc == -INFINITY) continue;
    const float w = expf(mc - M);
    l = fmaf(lc, w, l);
    o = fmaf(oc, w, o);
  }
  g[(size_t)r * H * Dh + h * Dh + e] = from_f<T>(o / l);
}

static int max_rows(const SeqRows& sr) {
  int m = 0;
  for (int b = 0; b < sr.nseq; ++b) m = std::max(m, sr.row0[b + 1] - sr.row0[b]);
  return m;
}

template <typename T, typename Src>
cudaError_t fir_dispatch(const LaunchCtx& L, Src s, int d, const SeqRows& sr, int Lf, int R, const float* taps,
                         const SeqPtrs<float*>& rings, const SeqPtrs<const evs_book*>& book, void* g) {
  const int NW = std::min(8, Lf);
  int J = 1;
  while (J * NW < Lf) J <<= 1;  // taps per warp, a power of two <= 32 (Lf <= 256)
  const int n = max_rows(sr);
  const size_t smem = sizeof(float) * 32 * ((Lf - 1 + n) + n + Lf + NW * n);
  void (*k)(Src, int, int, int, const float*, SeqRows, SeqPtrs<float*>, SeqPtrs<const evs_book*>, T*);
  switch (J) {
    case 1: k = fir_kernel<T, Src, 1>; break;
    case 2: k = fir_kernel<T, Src, 2>; break;
    case 4: k = fir_kernel<T, Src, 4>; break;
    case 8: k = fir_kernel<T, Src, 8>; break;
    case 16: k = fir_kernel<T, Src, 16>; break;
    case 32: k = fir_kernel<T, Src, 32>; break;
    default: return cudaErrorInvalidValue;
  }
  if (R < Lf - 1 + n) return cudaErrorInvalidValue;  // the window and the block must not alias
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  return launch(L, k, dim3(d / 32, sr.nseq), dim3(32 * NW), smem, s, d, Lf, R, taps, sr, rings, book, (T*)g);
}

template <typename T, typename Src, int M>
cudaError_t iir_dispatch_m(const LaunchCtx& L, Src s, int d, const SeqRows& sr, const float* lam, const float* res,
                           const SeqPtrs<float*>& s0, const SeqPtrs<float*>& s1,
                           const SeqPtrs<const evs_book*>& book, void* g) {
  constexpr int CPB = 256 / M;
  SeqPtrs<float2*> a{}, b{};
  for (int q = 0; q < sr.nseq; ++q) {
    a.p[q] = (float2*)s0.p[q];
    b.p[q] = (float2*)s1.p[q];
  }
  return launch(L, iir_kernel<T, Src, M>, dim3(d / CPB, sr.nseq), dim3(256), 0, s, d, (const float2*)lam,
                (const float2*)res, sr, a, b, book, (T*)g);
}

template <typename T, typename Src>
cudaError_t iir_dispatch(const LaunchCtx& L, Src s, int d, const SeqRows& sr, int M, const float* lam,
                         const float* res, const SeqPtrs<float*>& s0, const SeqPtrs<float*>& s1,
                         const SeqPtrs<const evs_book*>& book, void* g) {
  switch (M) {
    case 1: return iir_dispatch_m<T, Src, 1>(L, s, d, sr, lam, res, s0, s1, book, g);
    case 2: return iir_dispatch_m<T, Src, 2>(L, s, d, sr, lam, res, s0, s1, book, g);
    case 4: return iir_dispatch_m<T, Src, 4>(L, s, d, sr, lam, res, s0, s1, book, g);
    case 8: return iir_dispatch_m<T, Src, 8>(L, s, d, sr, lam, res, s0, s1, book, g);
    case 16: return iir_dispatch_m<T, Src, 16>(L, s, d, sr, lam, res, s0, s1, book, g);
    case 32: return iir_dispatch_m<T, Src, 32>(L, s, d, sr, lam, res, s0, s1, book, g);
    default: return cudaErrorInvalidValue;
  }
}

template <typename P, typename Q>
SeqPtrs<P> cast_ptrs(const SeqPtrs<Q>& in, int nseq) {
  SeqPtrs<P> out{};
  for (int b = 0; b < nseq; ++b) out.p[b] = (P)in.p[b];
  return out;
}

template <typename T, int DH, int CH>
cudaError_t attn_split_launch(const LaunchCtx& L, int H, const SeqRows& sr, long long ctx_max, const AttnSeq& as,
                              const AttnBufs& B) {
  const size_t smem = sizeof(float) * (NTOK * DH + NTOK * CH + NTOK * 4) +
                      (size_t)CH * (DH * sizeof(T) + 16) + (size_t)CH * DH * sizeof(T);
  auto k = attn_split_kernel<T, DH, CH>;
  static bool attr_set = false;
  if (!attr_set && smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  return launch(L, k, dim3(B.nsplit_max, H, sr.nseq), dim3(256), smem, (const float*)B.qbuf,
                cast_ptrs<const T*>(as.kc, sr.nseq), cast_ptrs<const T*>(as.vc, sr.nseq), H, sr, ctx_max,
                cast_ptrs<const evs_book*>(as.book, sr.nseq), B.span, as.part_o, as.part_ml, B.nsplit_max);
}

template <typename T, int DH>
cudaError_t attn_split_dispatch(const LaunchCtx& L, int H, const SeqRows& sr, long long ctx_max, int chunk,
                                const AttnSeq& as, const AttnBufs& B) {
  switch (chunk) {
    case 32: return attn_split_launch<T, DH, 32>(L, H, sr, ctx_max, as, B);
    case 64: return attn_split_launch<T, DH, 64>(L, H, sr, ctx_max, as, B);
    case 128: return attn_split_launch<T, DH, 128>(L, H, sr, ctx_max, as, B);
    case 256: return attn_split_launch<T, DH, 256>(L, H, sr, ctx_max, as, B);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T>
cudaError_t combine_launch(const LaunchCtx& L, int H, int Dh, const SeqRows& sr, long long ctx_max, const AttnSeq& as,
                           const AttnBufs& B, void* g) {
  const int rows = sr.row0[sr.nseq];
  return launch(L, attn_combine_kernel<T>, dim3(rows, H), dim3(Dh), 0, cast_ptrs<const float*>(as.part_o, sr.nseq),
                cast_ptrs<const float*>(as.part_ml, sr.nseq), H, Dh, sr, B.span, ctx_max,
                cast_ptrs<const evs_book*>(as.book, sr.nseq), B.nsplit_max, (T*)g);
}

template <typename T, typename Src>
cudaError_t attention_t(const LaunchCtx& L, Src s, int H, int Dh, const SeqRows& sr, long long ctx_max, int chunk,
                        const AttnSeq& as, const AttnBufs& B, void* g) {
  const int rows = sr.row0[sr.nseq];
  cudaError_t e = launch(L, qkv_rope_kernel<T, Src>, dim3(rows, H), dim3(Dh / 2), 0, s, H, Dh, ctx_max,
                         (const uint64_t*)B.turn_fx, sr, cast_ptrs<T*>(as.kc, sr.nseq), cast_ptrs<T*>(as.vc, sr.nseq),
                         B.qbuf, as.book);
  if (e != cudaSuccess) return e;
  switch (Dh) {
    case 32: e = attn_split_dispatch<T, 32>(L, H, sr, ctx_max, chunk, as, B); break;
    case 64: e = attn_split_dispatch<T, 64>(L, H, sr, ctx_max, chunk, as, B); break;
    case 128: e = attn_split_dispatch<T, 128>(L, H, sr, ctx_max, chunk, as, B); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  return combine_launch<T>(L, H, Dh, sr, ctx_max, as, B, g);
}

}  // namespace

cudaError_t launch_fir(const LaunchCtx& L, int dtype, MixSrc src, int d, const SeqRows& sr, int Lf, int R,
                       const float* taps, const SeqPtrs<float*>& rings, const SeqPtrs<const evs_book*>& book,
                       void* g) {
  const SrcPlain<float> sf{(const float*)src.p, src.ld};
  if (src.ws)
    return dtype == EVS_BF16 ? fir_dispatch<bf16>(L, SrcSlots{src.ws, src.tab, src.slot_rows}, d, sr, Lf, R, taps,
                                                  rings, book, g)
                             : cudaErrorInvalidValue;
  if (dtype == EVS_BF16)
    return src.f32 ? fir_dispatch<bf16>(L, sf, d, sr, Lf, R, taps, rings, book, g)
                   : fir_dispatch<bf16>(L, SrcPlain<bf16>{(const bf16*)src.p, src.ld}, d, sr, Lf, R, taps, rings,
                                        book, g);
  return fir_dispatch<float>(L, sf, d, sr, Lf, R, taps, rings, book, g);
}

cudaError_t launch_iir(const LaunchCtx& L, int dtype, MixSrc src, int d, const SeqRows& sr, int M,
                       const float* lam, const float* res, const SeqPtrs<float*>& st0, const SeqPtrs<float*>& st1,
                       const SeqPtrs<const evs_book*>& book, void* g) {
  const SrcPlain<float> sf{(const float*)src.p, src.ld};
  if (src.ws)
    return dtype == EVS_BF16 ? iir_dispatch<bf16>(L, SrcSlots{src.ws, src.tab, src.slot_rows}, d, sr, M, lam, res,
                                                  st0, st1, book, g)
                             : cudaErrorInvalidValue;
  if (dtype == EVS_BF16)
    return src.f32 ? iir_dispatch<bf16>(L, sf, d, sr, M, lam, res, st0, st1, book, g)
                   : iir_dispatch<bf16>(L, SrcPlain<bf16>{(const bf16*)src.p, src.ld}, d, sr, M, lam, res, st0,
                                        st1, book, g);
  return iir_dispatch<float>(L, sf, d, sr, M, lam, res, st0, st1, book, g);
}

// Key span of a split: max(chunk, 256) * 2^j, the smallest with at most
// ATTN_SPLITS_MAX splits over ctx_max.  Fixed per cache, so the partition
// of a query's keys never depends on the block size.
long long attn_span(long long ctx_max, int chunk) {
  long long span = std::max(chunk, 256);
  while ((ctx_max + span - 1) / span > ATTN_SPLITS_MAX) span *= 2;
  return span;
}

size_t attn_scratch_bytes(int H, int Dh, long long ctx_max, int chunk) {
  const long long nsplit = (ctx_max + attn_span(ctx_max, chunk) - 1) / attn_span(ctx_max, chunk);
  auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
  return al(sizeof(uint64_t) * (Dh / 2)) + al(sizeof(float) * ROWS_MAX * H * Dh) +
         al(sizeof(float) * H * nsplit * NTOK * Dh) + al(sizeof(float) * H * nsplit * NTOK * 2) +
         al(2 * sizeof(CUtensorMap)) + al(sizeof(int) * H);
}

void attn_bufs_from_scratch(void* scratch, int H, int Dh, long long ctx_max, int chunk, AttnBufs* out) {
  const long long span = attn_span(ctx_max, chunk);
  const long long nsplit = (ctx_max + span - 1) / span;
  auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
  char* p = (char*)scratch;
  out->turn_fx = (uint64_t*)p;
  p += al(sizeof(uint64_t) * (Dh / 2));
  out->qbuf = (float*)p;
  p += al(sizeof(float) * ROWS_MAX * H * Dh);
  out->part_o = (float*)p;
  p += al(sizeof(float) * H * nsplit * NTOK * Dh);
  out->part_ml = (float*)p;
  p += al(sizeof(float) * H * nsplit * NTOK * 2);
  out->maps = (CUtensorMap*)p;
  p += al(2 * sizeof(CUtensorMap));
  out->arrivals = (int*)p;
  out->nsplit_max = (int)nsplit;
  out->span = (int)span;
}

cudaError_t fill_rope_table(const AttnBufs& B, int Dh, float rope_base, cudaStream_t stream) {
  uint64_t fx[512];
  if (Dh / 2 > 512) return cudaErrorInvalidValue;
  const double TWO_PI = 6.283185307179586476925287;
  for (int i = 0; i < Dh / 2; ++i) {
    // turns per position base^(-2i/Dh) / (2 pi), scaled by 2^64 (below 2^64:
    // the frequency is at most 1 < 2 pi); a double carries it to 2^-53
    // relative, far below the float angle's resolution at any position
    // below 2^31
    const double f = std::pow((double)rope_base, -2.0 * (double)i / (double)Dh);
    fx[i] = (uint64_t)std::ldexp(f / TWO_PI, 64);
  }
  cudaError_t e = cudaMemcpyAsync(B.turn_fx, fx, sizeof(uint64_t) * (Dh / 2), cudaMemcpyHostToDevice, stream);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(stream);  // fx lives on this stack frame
}

cudaError_t launch_attention(const LaunchCtx& L, int dtype, MixSrc src, int H, int Dh, const SeqRows& sr,
                             long long ctx_max, int chunk, const AttnSeq& as, const AttnBufs& B, void* g) {
  if (attn_tma_eligible(dtype, H, Dh, ctx_max)) {
    if (ctx_max > ATTN_SHORT_CACHE)
      // long bf16 caches: rotary embedding, append, split-KV and the combine
      // in one kernel
      return launch_attn_tma(L, src, H, Dh, sr, ctx_max, as, B, g, true);
    // short ones: a few stages per split, all splits at once; the three
    // steps as separate kernels overlap better under dependent launch
    const int rows = sr.row0[sr.nseq];
    auto rope = [&](auto s) {
      return launch(L, qkv_rope_kernel<bf16, decltype(s)>, dim3(rows, H), dim3(Dh / 2), 0, s, H, Dh, ctx_max,
                    (const uint64_t*)B.turn_fx, sr, cast_ptrs<bf16*>(as.kc, sr.nseq),
                    cast_ptrs<bf16*>(as.vc, sr.nseq), B.qbuf, as.book);
    };
    cudaError_t e = src.ws ? rope(SrcSlots{src.ws, src.tab, src.slot_rows})
                           : src.f32 ? rope(SrcPlain<float>{(const float*)src.p, src.ld})
                                     : rope(SrcPlain<bf16>{(const bf16*)src.p, src.ld});
    if (e != cudaSuccess) return e;
    e = launch_attn_tma(L, src, H, Dh, sr, ctx_max, as, B, g, false);
    if (e != cudaSuccess) return e;
    return combine_launch<bf16>(L, H, Dh, sr, ctx_max, as, B, g);
  }
  const SrcPlain<float> sf{(const float*)src.p, src.ld};
  if (src.ws)
    return dtype == EVS_BF16 ? attention_t<bf16>(L, SrcSlots{src.ws, src.tab, src.slot_rows}, H, Dh, sr, ctx_max,
                                                 chunk, as, B, g)
                             : cudaErrorInvalidValue;
  if (dtype == EVS_BF16)
    return src.f32 ? attention_t<bf16>(L, sf, H, Dh, sr, ctx_max, chunk, as, B, g)
                   : attention_t<bf16>(L, SrcPlain<bf16>{(const bf16*)src.p, src.ld}, H, Dh, sr, ctx_max, chunk, as,
                                       B, g);
  return attention_t<float>(L, sf, H, Dh, sr, ctx_max, chunk, as, B, g);
}

}  // namespace evs
