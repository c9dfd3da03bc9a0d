// Sequence mixers of the hybrid stack for one verify block, each keeping the
// state after every block position ("What we implemented" in the EvSpark
// discussion post; author's reply, prerequisite 1):
//
//  FIR  (short / medium Hyena filter): the window of the last L-1 inputs and
//       the block's n new inputs form one "ext" buffer [L-1+n][d]; position
//       i's window is ext rows [i+1, i+L).  The kernel writes ext to the
//       spare bank, so commit only moves an offset.
//  IIR  (modal Hyena filter): s_t = lam * s_{t-1} + z_t per channel and pole,
//       y_t = Re sum_m R_m s_t[m]; all n states go to the spare bank.
//  ATTN rotary q/k, append k/v at rows pos..pos+n-1 (append-only cache),
//       split-KV block-causal attention with a fixed-order combine.
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
// registers.
template <typename T, typename Src, int JT>
__global__ void __launch_bounds__(256) fir_kernel(Src src, int d, int n, int Lf,
                                                  const float* __restrict__ taps, float* ext0,
                                                  float* ext1, const evs_book* book, T* g) {
  extern __shared__ float sm[];
  const int NW = blockDim.x >> 5;
  const int rows = Lf - 1 + n;
  float* ext_s = sm;                       // [rows][32]
  float* a_s = ext_s + rows * 32;          // [n][32]
  float* tap_s = a_s + n * 32;             // [Lf][32]
  float* part_s = tap_s + Lf * 32;         // [NW][n][32]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c0 = blockIdx.x * 32, c = c0 + lane;

  pdl_trigger();
  // Taps, the committed window and its copy into the spare bank do not
  // depend on the in-projection: done while the preceding GEMM still runs
  // (the bank / offset are fixed for the whole verify).
  const int bank = book->fir_bank, off = book->fir_off;
  const float* src_ext = bank ? ext1 : ext0;
  float* dst_ext = bank ? ext0 : ext1;
  // rows of 32 channels = 128 bytes = 8 x 16-byte pieces, all copies in flight at once
  const int nthr = blockDim.x;
  for (int e = threadIdx.x; e < Lf * 8; e += nthr) {
    const int j = e >> 3, w = e & 7;
    cp_async16(tap_s + j * 32 + w * 4, taps + (size_t)j * d + c0 + w * 4);
  }
  for (int e = threadIdx.x; e < (Lf - 1) * 8; e += nthr) {
    const int r = e >> 3, w = e & 7;
    cp_async16(ext_s + r * 32 + w * 4, src_ext + (size_t)(off + r) * d + c0 + w * 4);
  }
  cp_async_wait_all();
  __syncthreads();
  for (int e = threadIdx.x; e < (Lf - 1) * 8; e += nthr) {
    const int r = e >> 3, w = e & 7;
    *reinterpret_cast<float4*>(dst_ext + (size_t)r * d + c0 + w * 4) =
        *reinterpret_cast<const float4*>(ext_s + r * 32 + w * 4);
  }
  pdl_wait();
  for (int t = warp; t < n; t += NW) {
    const float a = stored<T>(src.get(t, c));
    const float b = stored<T>(src.get(t, d + c));
    const float v = stored<T>(src.get(t, 2 * d + c));
    a_s[t * 32 + lane] = a;
    ext_s[(Lf - 1 + t) * 32 + lane] = b * v;
    dst_ext[(size_t)(Lf - 1 + t) * d + c] = b * v;
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
#pragma unroll
  for (int t = 0; t < NTOK; ++t) {
    if (t < n) {
      float acc = 0.f;
#pragma unroll
      for (int q = 0; q < JT; ++q)
        if (j0 + q < Lf) acc = fmaf(hreg[q], wreg[t - q + JT - 1], acc);
      part_s[(warp * n + t) * 32 + lane] = acc;
    }
  }
  __syncthreads();
  for (int t = warp; t < n; t += NW) {
    float y = 0.f;
    for (int w = 0; w < NW; ++w) y += part_s[(w * n + t) * 32 + lane];
    g[(size_t)t * d + c] = from_f<T>(a_s[t * 32 + lane] * y);
  }
}

// ------------------------------------------------------------------ IIR
// Block = 256 threads = (256/M) channels x M poles, poles of a channel in
// adjacent lanes.  Per-position states land in the spare bank [n][d][M].
template <typename T, typename Src, int M>
__global__ void __launch_bounds__(256) iir_kernel(Src src, int d, int n, const float2* __restrict__ lam,
                                                  const float2* __restrict__ res, float2* st0,
                                                  float2* st1, const evs_book* book, T* g) {
  constexpr int CPB = 256 / M;
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
  pdl_wait();
  for (int e = threadIdx.x; e < n * CPB; e += 256) {
    const int t = e / CPB, cc = blockIdx.x * CPB + e % CPB;
    const float a = stored<T>(src.get(t, cc));
    const float b = stored<T>(src.get(t, d + cc));
    const float v = stored<T>(src.get(t, 2 * d + cc));
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
    if (m == 0) g[(size_t)t * d + c] = from_f<T>(a_s[t][cl] * y);
  }
}

// ------------------------------------------------------------------ attention
// (1) rotary embedding + append: grid (n, H), Dh/2 threads, one rotation pair each.
template <typename T, typename Src>
__global__ void qkv_rope_kernel(Src src, int H, int Dh, int n, long long ctx_max, const double* inv_freq, T* kc,
                                T* vc, float* qbuf, evs_book* book) {
  const int t = blockIdx.x, h = blockIdx.y, i = threadIdx.x, half = Dh >> 1;
  const int d = H * Dh;
  pdl_trigger();
  // the position is fixed for the whole verify: the rotation is computed
  // while the in-projection still runs.  Angle pos * base^(-2i/Dh) in
  // double (table built on the host in double), reduced to [-pi, pi] in
  // double, then sin / cos in float.
  const long long pos = (long long)book->pos + t;
  const double TWO_PI = 6.283185307179586476925287;
  const double ang = (double)pos * inv_freq[i];
  const double turns = rint(ang * (1.0 / TWO_PI));
  const float red = (float)fma(-turns, TWO_PI, ang);
  float sn, cs;
  sincosf(red, &sn, &cs);
  pdl_wait();
  if (pos >= ctx_max) {
    if (i == 0) set_status(book, EVS_DEV_KV_OVERFLOW);
    return;
  }
  const int col = h * Dh + i;
  const float q1 = stored<T>(src.get(t, col)), q2 = stored<T>(src.get(t, col + half));
  const float k1 = stored<T>(src.get(t, d + col)), k2 = stored<T>(src.get(t, d + col + half));
  const float v1 = stored<T>(src.get(t, 2 * d + col)), v2 = stored<T>(src.get(t, 2 * d + col + half));
  const float rq1 = q1 * cs - q2 * sn, rq2 = q1 * sn + q2 * cs;
  const float rk1 = k1 * cs - k2 * sn, rk2 = k1 * sn + k2 * cs;
  const size_t row = ((size_t)h * ctx_max + pos) * Dh;
  kc[row + i] = from_f<T>(rk1);
  kc[row + i + half] = from_f<T>(rk2);
  vc[row + i] = from_f<T>(v1);
  vc[row + i + half] = from_f<T>(v2);
  float* qo = qbuf + ((size_t)t * H + h) * Dh;
  qo[i] = stored<T>(rq1);
  qo[i + half] = stored<T>(rq2);
}

// (2) split-KV: CTA (x, h) handles chunks x, x+gridDim.x, ... of CH keys
// at absolute positions [cidx*CH, (cidx+1)*CH).  Query t (position pos+t)
// sees keys <= pos+t.  Each chunk's K and V rows are staged in shared
// memory (K rows padded by 16 bytes so the per-key dot products of a warp
// hit distinct banks); per chunk and query the kernel stores the max, the
// sum of exp and the unnormalised output.  Every reduction runs over fixed
// key slots, masked slots contributing exact zeros, so a query's result does
// not depend on the other queries of the block.
template <typename T, int DH, int CH>
__global__ void __launch_bounds__(256) attn_split_kernel(const float* __restrict__ qbuf, const T* __restrict__ kc,
                                                         const T* __restrict__ vc, int H, int n,
                                                         long long ctx_max, const evs_book* book, float* part_o,
                                                         float* part_ml, int nchunk_max) {
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
  float* ml_s = p_s + NTOK * CH;                                   // [NTOK][2]
  unsigned char* k_s = reinterpret_cast<unsigned char*>(ml_s + NTOK * 2);  // [CH][KP]
  unsigned char* v_s = k_s + CH * KP;                              // [CH][VP]
  const int h = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_trigger();
  // the committed length is fixed for the whole verify: pull this CTA's
  // committed keys / values into L2 while the in-projection still runs
  const long long pos = book->pos;
  const long long total = min(pos + n, ctx_max);
  const int nchunks = (int)((total + CH - 1) / CH);
  if (tid == 0) {
    for (int cidx = blockIdx.x; cidx < nchunks; cidx += gridDim.x) {
      const long long k0 = (long long)cidx * CH;
      const long long nk = min((long long)CH, min(pos, ctx_max) - k0);
      if (nk > 0) {
        const unsigned bytes = (unsigned)(nk * DH * sizeof(T));
        const T* kr = kc + ((size_t)h * ctx_max + k0) * DH;
        const T* vr = vc + ((size_t)h * ctx_max + k0) * DH;
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(kr), "r"(bytes) : "memory");
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(vr), "r"(bytes) : "memory");
      }
    }
  }
  pdl_wait();
  const float scale = rsqrtf((float)DH);
  for (int e = tid; e < NTOK * DH; e += 256) {
    const int t = e / DH;
    q_s[e] = t < n ? qbuf[((size_t)t * H + h) * DH + e % DH] : 0.f;
  }
  for (int cidx = blockIdx.x; cidx < nchunks; cidx += gridDim.x) {
    const long long k0 = (long long)cidx * CH;
    const int kmax = (int)min((long long)CH, total - k0);
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
    // per query: max and sum of exp over the chunk's slots (warp per query)
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
        ml_s[t * 2] = mx;
        ml_s[t * 2 + 1] = sum;
      }
    }
    __syncthreads();
    // unnormalised output: thread = (dim pair dp, query group tq)
    {
      const int dp = tid % DP, tq = tid / DP;
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
          const int t = tq + r * OG;
          if (t < n) {
            const float p = p_s[t * CH + j];
            o0[r] = fmaf(p, v0, o0[r]);
            o1[r] = fmaf(p, v1, o1[r]);
          }
        }
      }
#pragma unroll
      for (int r = 0; r < OS; ++r) {
        const int t = tq + r * OG;
        if (t < n) {
          float* o = part_o + (((size_t)h * nchunk_max + cidx) * NTOK + t) * DH + 2 * dp;
          o[0] = o0[r];
          o[1] = o1[r];
        }
      }
    }
    if (tid < n) {
      float* ml = part_ml + (((size_t)h * nchunk_max + cidx) * NTOK + tid) * 2;
      ml[0] = ml_s[tid * 2];
      ml[1] = ml_s[tid * 2 + 1];
    }
  }
}

// (3) combine: grid (n, H), Dh threads; chunks in ascending order.
template <typename T>
__global__ void attn_combine_kernel(const float* part_o, const float* part_ml, int H, int Dh, int n,
                                    int chunk, long long ctx_max, const evs_book* book, int nchunk_max, T* g) {
  const int t = blockIdx.x, h = blockIdx.y, e = threadIdx.x;
  pdl_trigger();
  pdl_wait();
  const long long qpos = min((long long)book->pos + t, ctx_max - 1);
  const int nc = (int)(qpos / chunk) + 1;  // chunks holding keys <= qpos
  const float* ml = part_ml + ((size_t)h * nchunk_max * NTOK + t) * 2;
  float M = -INFINITY;
#pragma unroll 8
  for (int c = 0; c < nc; ++c) M = fmaxf(M, ml[(size_t)c * NTOK * 2]);
  float l = 0.f, o = 0.f;
  // loads are independent of the running sums: unrolled so they overlap
#pragma unroll 8
  for (int c = 0; c < nc; ++c) {
    const float mc = ml[(size_t)c * NTOK * 2];
    const float lc = ml[(size_t)c * NTOK * 2 + 1];
    const float oc = part_o[(((size_t)h * nchunk_max + c) * NTOK + t) * Dh + e];
    if (mc == -INFINITY) continue;
    const float w = expf(mc - M);
    l = fmaf(lc, w, l);
    o = fmaf(oc, w, o);
  }
  g[(size_t)t * H * Dh + h * Dh + e] = from_f<T>(o / l);
}

template <typename T, typename Src>
cudaError_t fir_dispatch(const LaunchCtx& L, Src s, int d, int n, int Lf, const float* taps,
                         float* e0, float* e1, const evs_book* book, void* g) {
  const int NW = std::min(8, Lf);
  int J = 1;
  while (J * NW < Lf) J <<= 1;  // taps per warp, a power of two <= 32 (Lf <= 256)
  const size_t smem = sizeof(float) * 32 * ((Lf - 1 + n) + n + Lf + NW * n);
  void (*k)(Src, int, int, int, const float*, float*, float*, const evs_book*, T*);
  switch (J) {
    case 1: k = fir_kernel<T, Src, 1>; break;
    case 2: k = fir_kernel<T, Src, 2>; break;
    case 4: k = fir_kernel<T, Src, 4>; break;
    case 8: k = fir_kernel<T, Src, 8>; break;
    case 16: k = fir_kernel<T, Src, 16>; break;
    case 32: k = fir_kernel<T, Src, 32>; break;
    default: return cudaErrorInvalidValue;
  }
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  return launch(L, k, dim3(d / 32), dim3(32 * NW), smem, s, d, n, Lf, taps, e0, e1, book, (T*)g);
}

template <typename T, typename Src, int M>
cudaError_t iir_dispatch_m(const LaunchCtx& L, Src s, int d, int n, const float* lam, const float* res,
                           float* s0, float* s1, const evs_book* book, void* g) {
  constexpr int CPB = 256 / M;
  return launch(L, iir_kernel<T, Src, M>, dim3(d / CPB), dim3(256), 0, s, d, n,
                (const float2*)lam, (const float2*)res, (float2*)s0, (float2*)s1, book, (T*)g);
}

template <typename T, typename Src>
cudaError_t iir_dispatch(const LaunchCtx& L, Src s, int d, int n, int M, const float* lam,
                         const float* res, float* s0, float* s1, const evs_book* book, void* g) {
  switch (M) {
    case 1: return iir_dispatch_m<T, Src, 1>(L, s, d, n, lam, res, s0, s1, book, g);
    case 2: return iir_dispatch_m<T, Src, 2>(L, s, d, n, lam, res, s0, s1, book, g);
    case 4: return iir_dispatch_m<T, Src, 4>(L, s, d, n, lam, res, s0, s1, book, g);
    case 8: return iir_dispatch_m<T, Src, 8>(L, s, d, n, lam, res, s0, s1, book, g);
    case 16: return iir_dispatch_m<T, Src, 16>(L, s, d, n, lam, res, s0, s1, book, g);
    case 32: return iir_dispatch_m<T, Src, 32>(L, s, d, n, lam, res, s0, s1, book, g);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T, int DH, int CH>
cudaError_t attn_split_launch(const LaunchCtx& L, int H, int n, long long ctx_max, evs_book* book,
                              const AttnBufs& B, void* kc, void* vc, int num_sms) {
  const size_t smem = sizeof(float) * (NTOK * DH + NTOK * CH + NTOK * 2) +
                      (size_t)CH * (DH * sizeof(T) + 16) + (size_t)CH * DH * sizeof(T);
  auto k = attn_split_kernel<T, DH, CH>;
  static bool attr_set = false;
  if (!attr_set && smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int gx = std::max(1, std::min(B.nchunk_max, (4 * num_sms + H - 1) / H));
  return launch(L, k, dim3(gx, H), dim3(256), smem, (const float*)B.qbuf, (const T*)kc, (const T*)vc, H, n,
                ctx_max, (const evs_book*)book, B.part_o, B.part_ml, B.nchunk_max);
}

template <typename T, int DH>
cudaError_t attn_split_dispatch(const LaunchCtx& L, int H, int n, long long ctx_max, int chunk,
                                evs_book* book, const AttnBufs& B, void* kc, void* vc, int num_sms) {
  switch (chunk) {
    case 32: return attn_split_launch<T, DH, 32>(L, H, n, ctx_max, book, B, kc, vc, num_sms);
    case 64: return attn_split_launch<T, DH, 64>(L, H, n, ctx_max, book, B, kc, vc, num_sms);
    case 128: return attn_split_launch<T, DH, 128>(L, H, n, ctx_max, book, B, kc, vc, num_sms);
    case 256: return attn_split_launch<T, DH, 256>(L, H, n, ctx_max, book, B, kc, vc, num_sms);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T, typename Src>
cudaError_t attention_t(const LaunchCtx& L, Src s, int H, int Dh, int n, long long ctx_max, int chunk,
                        void* kc, void* vc, evs_book* book, const AttnBufs& B, void* g, int num_sms) {
  cudaError_t e = launch(L, qkv_rope_kernel<T, Src>, dim3(n, H), dim3(Dh / 2), 0, s, H, Dh, n, ctx_max,
                         (const double*)B.inv_freq, (T*)kc, (T*)vc, B.qbuf, book);
  if (e != cudaSuccess) return e;
  switch (Dh) {
    case 32: e = attn_split_dispatch<T, 32>(L, H, n, ctx_max, chunk, book, B, kc, vc, num_sms); break;
    case 64: e = attn_split_dispatch<T, 64>(L, H, n, ctx_max, chunk, book, B, kc, vc, num_sms); break;
    case 128: e = attn_split_dispatch<T, 128>(L, H, n, ctx_max, chunk, book, B, kc, vc, num_sms); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  return launch(L, attn_combine_kernel<T>, dim3(n, H), dim3(Dh), 0, (const float*)B.part_o,
                (const float*)B.part_ml, H, Dh, n, chunk, ctx_max, (const evs_book*)book, B.nchunk_max, (T*)g);
}

}  // namespace

cudaError_t launch_fir(const LaunchCtx& L, int dtype, MixSrc src, int d, int n, int Lf, const float* taps,
                       float* ext0, float* ext1, const evs_book* book, void* g) {
  const SrcPlain<float> sf{(const float*)src.p, src.ld};
  if (dtype == EVS_BF16)
    return src.f32 ? fir_dispatch<bf16>(L, sf, d, n, Lf, taps, ext0, ext1, book, g)
                   : fir_dispatch<bf16>(L, SrcPlain<bf16>{(const bf16*)src.p, src.ld}, d, n, Lf, taps, ext0,
                                        ext1, book, g);
  return fir_dispatch<float>(L, sf, d, n, Lf, taps, ext0, ext1, book, g);
}

cudaError_t launch_iir(const LaunchCtx& L, int dtype, MixSrc src, int d, int n, int M, const float* lam,
                       const float* res, float* st0, float* st1, const evs_book* book, void* g) {
  const SrcPlain<float> sf{(const float*)src.p, src.ld};
  if (dtype == EVS_BF16)
    return src.f32 ? iir_dispatch<bf16>(L, sf, d, n, M, lam, res, st0, st1, book, g)
                   : iir_dispatch<bf16>(L, SrcPlain<bf16>{(const bf16*)src.p, src.ld}, d, n, M, lam, res, st0,
                                        st1, book, g);
  return iir_dispatch<float>(L, sf, d, n, M, lam, res, st0, st1, book, g);
}

size_t attn_scratch_bytes(int H, int Dh, long long ctx_max, int chunk) {
  const long long nchunk = (ctx_max + chunk - 1) / chunk;
  auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
  return al(sizeof(double) * (Dh / 2)) + al(sizeof(float) * NTOK * H * Dh) +
         al(sizeof(float) * H * nchunk * NTOK * Dh) + al(sizeof(float) * H * nchunk * NTOK * 2);
}

void attn_bufs_from_scratch(void* scratch, int H, int Dh, long long ctx_max, int chunk, AttnBufs* out) {
  const long long nchunk = (ctx_max + chunk - 1) / chunk;
  auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
  char* p = (char*)scratch;
  out->inv_freq = (double*)p;
  p += al(sizeof(double) * (Dh / 2));
  out->qbuf = (float*)p;
  p += al(sizeof(float) * NTOK * H * Dh);
  out->part_o = (float*)p;
  p += al(sizeof(float) * H * nchunk * NTOK * Dh);
  out->part_ml = (float*)p;
  out->nchunk_max = (int)nchunk;
}

cudaError_t fill_rope_table(const AttnBufs& B, int Dh, float rope_base, cudaStream_t stream) {
  double tab[512];
  if (Dh / 2 > 512) return cudaErrorInvalidValue;
  for (int i = 0; i < Dh / 2; ++i) tab[i] = std::pow((double)rope_base, -2.0 * (double)i / (double)Dh);
  cudaError_t e = cudaMemcpyAsync(B.inv_freq, tab, sizeof(double) * (Dh / 2), cudaMemcpyHostToDevice, stream);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(stream);  // tab lives on this stack frame
}

cudaError_t launch_attention(const LaunchCtx& L, int dtype, MixSrc src, int H, int Dh, int n,
                             long long ctx_max, int chunk, void* kc, void* vc,
                             evs_book* book, const AttnBufs& B, void* g, int num_sms) {
  const SrcPlain<float> sf{(const float*)src.p, src.ld};
  if (dtype == EVS_BF16)
    return src.f32 ? attention_t<bf16>(L, sf, H, Dh, n, ctx_max, chunk, kc, vc, book, B, g, num_sms)
                   : attention_t<bf16>(L, SrcPlain<bf16>{(const bf16*)src.p, src.ld}, H, Dh, n, ctx_max, chunk,
                                       kc, vc, book, B, g, num_sms);
  return attention_t<float>(L, sf, H, Dh, n, ctx_max, chunk, kc, vc, book, B, g, num_sms);
}

}  // namespace evs
