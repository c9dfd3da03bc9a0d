// Persistent verify engine: one kernel per span of the verify step between
// attention mixers (see EngPhase in evs_internal.cuh).
//
// The verify step is bound by the weight read (the discussion post's reply,
// "Regime overlap").  Run as separate kernels, every layer boundary stops
// the weight stream: the GEMM drains, the small kernel between two GEMMs
// waits for it to finish, and the next GEMM waits for the small kernel.
// Here each CTA (one per SM) keeps streaming its share of the next weight
// matrices into a shared-memory ring while the row work between GEMMs runs
// on other warps; only the tensor-core MMA waits for activations.
//
// Warp roles of a CTA (512 threads):
//   0      weight producer: one bulk copy per 16 KB packed unit into the ring,
//          in the order the GEMM phases follow each other, plus an L2
//          prefetch window E_PF units further ahead; waits only for ring
//          slots
//   1      MMA issuer: tcgen05.mma of each unit into a 128 x 16 fp32 TMEM
//          accumulator (double-buffered per tile segment)
//   2      activation loader: before a GEMM phase's first unit, waits until
//          the phase that writes its activations has counted all its items,
//          then fetches the 2 KB activation tile of every unit by TMA
//   4..7   epilogue: TMEM -> the tile's partial slot, then counts the tile
//   8..15  row work: FIR / IIR mixers, residual add + sums of squares,
//          RMSNorm, SiLU-and-multiply, logits; items spread over the CTAs
// Every wait is bounded: a wait that runs out raises a CTA flag and a
// global flag that every other wait polls, each role then leaves its loop,
// in-flight copies and MMAs are waited for, TMEM is freed and the kernel
// returns with EVS_DEV_TIMEOUT in the state's status.
#include "evs_internal.cuh"
#include "ptx.cuh"

namespace evs {
namespace {

constexpr int E_S = 8;             // ring stages (weight + activation tile each)
constexpr int E_SLOG = 3;          // log2(E_S)
static_assert((1 << E_SLOG) == E_S, "ring depth is a power of two");
constexpr int E_PF = 16;           // units kept prefetched into L2 beyond the ring
constexpr int E_THREADS = 512;
constexpr int E_EPI0 = 4;          // first epilogue warp (warps 4..7 own TMEM lane quarters 0..3)
constexpr int E_ROW0 = 8;          // first row-work warp
constexpr int E_ROWW = 8;          // row-work warps
constexpr int E_ROWT = E_ROWW * 32;
constexpr int EA_BYTES = TILE_M * TILE_K * 2;  // 16 KB weight unit
constexpr int EB_BYTES = NTOK * TILE_K * 2;    // 2 KB activation tile
constexpr uint64_t E_WAIT_NS = 2000000000ull;  // bound on any wait
// [1 KB alignment slack][ring A][ring B][barriers][flags][row-work area, 128-byte aligned]
constexpr size_t E_BAR_OFF = (size_t)E_S * (EA_BYTES + EB_BYTES);
constexpr size_t E_ROW_OFF = (E_BAR_OFF + (3 * E_S + 5) * 8 + 64 + 127) & ~(size_t)127;
constexpr size_t E_FIXED = 1024 + E_ROW_OFF;

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void red_release_add(int* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// generic-proxy writes of this thread -> later async-proxy (TMA) reads
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(smem_dst)),
               "l"(gmem_src)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ void row_sync() { asm volatile("bar.sync 3, %0;" ::"n"(E_ROWT) : "memory"); }
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

struct Abort {
  volatile int* local;   // this CTA
  volatile int* global;  // the launch
};
__device__ __forceinline__ bool aborted(const Abort& ab) { return *ab.local || *ab.global; }
__device__ __noinline__ void raise_abort(const Abort& ab) {
  *ab.local = 1;
  atomicExch((int*)ab.global, 1);
}

// Bounded mbarrier wait: false once the bound passes (both flags raised) or
// another wait has already given up.
__device__ __noinline__ bool e_mbar_wait_slow(uint32_t bar, uint32_t parity, Abort ab) {
  const uint64_t t0 = gtimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try(bar, parity)) return true;
    if ((i & 31) == 0) {
      if (aborted(ab)) return false;
      if (gtimer() - t0 > E_WAIT_NS) {
        raise_abort(ab);
        return false;
      }
    }
  }
}
__device__ __forceinline__ bool e_mbar_wait(uint32_t bar, uint32_t parity, Abort ab) {
  return mbar_try(bar, parity) || e_mbar_wait_slow(bar, parity, ab);
}
// Bounded wait until the counter reaches target (acquire).
__device__ __noinline__ bool e_count_wait_slow(const int* p, int target, Abort ab) {
  const uint64_t t0 = gtimer();
  for (uint32_t i = 1;; ++i) {
    if (ld_acquire(p) >= target) return true;
    if ((i & 7) == 0) {
      if (aborted(ab)) return false;
      if (gtimer() - t0 > E_WAIT_NS) {
        raise_abort(ab);
        return false;
      }
    }
    __nanosleep(64);
  }
}
__device__ __forceinline__ bool e_count_wait(const int* p, int target, Abort ab) {
  return ld_acquire(p) >= target || e_count_wait_slow(p, target, ab);
}
// Wait for copies already issued into this CTA's shared memory (teardown
// after an abort: the CTA must not exit with a copy in flight).
__device__ void drain_wait(uint32_t bar, uint32_t parity) {
  volatile int own = 0;
  mbar_wait_slow(bar, parity, &own);
}

// This CTA's unit range [ub, ue) of a GEMM phase (empty if it takes no part).
__device__ __forceinline__ void unit_range(const EngPhase& P, int c, long long* ub, long long* ue) {
  if (c < P.G) {
    *ub = unit_begin(P.U, P.G, c);
    *ue = unit_begin(P.U, P.G, c + 1);
  } else {
    *ub = *ue = 0;
  }
}

// ------------------------------------------------------------------ row work
// Items of the row phases.  Each is done by the 256 row-work threads of one
// CTA (rt = their index); the arithmetic and its order are those of the
// separate kernels (mixers.cu, rowops.cu), so the results are the same bits.

// Waits (one thread) until every contributor of the listed tiles of the
// GEMM whose slots a row phase reads has finished; the row threads proceed
// together.

__device__ bool row_wait_tiles(const EngPhase& P, const int* tiles, int k, Abort ab, volatile int* s_flag) {
  const int rt = threadIdx.x - E_ROW0 * 32;
  if (rt == 0) {
    bool ok = true;
    for (int i = 0; i < k && ok; ++i) ok = e_count_wait(P.cnt + tiles[i], __ldg(&P.tab[tiles[i]].y), ab);
    *s_flag = ok ? 1 : 0;
  }
  row_sync();
  const bool ok = *s_flag != 0;
  row_sync();  // the flag is read by all before its next use
  return ok;
}
// All row threads' outputs of an item are written: make them visible to the
// async proxy (TMA readers), then count the item.
__device__ void row_signal(int* counter, bool tma_readers) {
  if (tma_readers) fence_proxy_async_global();
  row_sync();
  if (threadIdx.x == E_ROW0 * 32) {
    red_release_add(counter, 1);
  }
}

// FIR mixer for 32 channels (fir_kernel's arithmetic; the taps are split
// over min(8, L) warps of JT taps).
template <int JT>
__device__ bool fir_item(const EngPhase& P, int j, int n, int d, const evs_book* book, float* sm, Abort ab,
                         volatile int* s_flag) {
  const int Lf = P.L, NW = min(8, Lf), rows = Lf - 1 + n;
  float* ext_s = sm;               // [rows][32]
  float* a_s = ext_s + rows * 32;  // [n][32]
  float* tap_s = a_s + n * 32;     // [Lf][32]
  float* part_s = tap_s + Lf * 32; // [NW][n][32]
  const int rt = threadIdx.x - E_ROW0 * 32, lane = rt & 31, warp = rt >> 5;
  const int c0 = j * 32, c = c0 + lane;
  // the ring: the input of position p at row p mod R (fir_kernel's layout)
  const long long pos = book->pos;
  const int R = P.ring;
  float* ring = P.bank0;
  bf16* g = static_cast<bf16*>(P.out);
  // taps and the committed window do not depend on the in-projection
  for (int e = rt; e < Lf * 8; e += E_ROWT) {
    const int q = e >> 3, w = e & 7;
    cp_async16(tap_s + q * 32 + w * 4, P.p0 + (size_t)q * d + c0 + w * 4);
  }
  for (int e = rt; e < (Lf - 1) * 8; e += E_ROWT) {
    const int r = e >> 3, w = e & 7;
    const long long p = pos - (Lf - 1) + r;  // rows before position 0 hold zeros
    const int pr = (int)(p >= 0 ? p % R : p + R);
    cp_async16(ext_s + r * 32 + w * 4, ring + (size_t)pr * d + c0 + w * 4);
  }
  cp_async_wait_all();
  row_sync();
  const int tiles[3] = {c0 / TILE_M, (d + c0) / TILE_M, (2 * d + c0) / TILE_M};
  if (!row_wait_tiles(P, tiles, 3, ab, s_flag)) return false;
  const SrcSlots src{P.ws, P.tab, NTOK};
  const auto ca = src.at(c), cb = src.at(d + c), cv = src.at(2 * d + c);
  for (int t0 = warp; t0 < n; t0 += 3 * E_ROWW) {
    float av[3], bv[3], vv[3];
#pragma unroll
    for (int k = 0; k < 3; ++k) {
      const int t = min(t0 + k * E_ROWW, n - 1);
      av[k] = src.get(ca, t, c);
      bv[k] = src.get(cb, t, d + c);
      vv[k] = src.get(cv, t, 2 * d + c);
    }
#pragma unroll
    for (int k = 0; k < 3; ++k) {
      const int t = t0 + k * E_ROWW;
      if (t < n) {
        const float a = stored<bf16>(av[k]), b = stored<bf16>(bv[k]), v = stored<bf16>(vv[k]);
        a_s[t * 32 + lane] = a;
        ext_s[(Lf - 1 + t) * 32 + lane] = b * v;
        ring[(size_t)((pos + t) % R) * d + c] = b * v;
      }
    }
  }
  row_sync();
  if (warp < NW) {
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
  }
  row_sync();
  for (int t = warp; t < n; t += E_ROWW) {
    float y = 0.f;
    for (int w = 0; w < NW; ++w) y += part_s[(w * n + t) * 32 + lane];
    g[(size_t)t * d + c] = __float2bfloat16_rn(a_s[t * 32 + lane] * y);
  }
  row_signal(P.ready, true);
  row_sync();  // shared memory is reused by the next item
  return true;
}

// IIR modal mixer for NS blocks of 256 / M channels (iir_kernel's
// arithmetic); thread (cl, m) runs pole m of channel cl of every block, the
// blocks' recurrences interleaved.
template <int M, int NS>
__device__ bool iir_item(const EngPhase& P, int j, int n, int d, const evs_book* book, float* sm, Abort ab,
                         volatile int* s_flag) {
  constexpr int CPB = 256 / M, CH = NS * CPB;
  float* z_s = sm;             // [NTOK][CH]
  float* a_s = sm + NTOK * CH; // [NTOK][CH]
  const int rt = threadIdx.x - E_ROW0 * 32;
  const int cl = rt / M, m = rt % M;
  const int c0 = j * CH;
  const float2* lam = reinterpret_cast<const float2*>(P.p0);
  const float2* res = reinterpret_cast<const float2*>(P.p1);
  const int bank = book->iir_bank, slot = book->iir_slot;
  const float2* cur = reinterpret_cast<const float2*>(bank ? P.bank1 : P.bank0);
  float2* dst = reinterpret_cast<float2*>(bank ? P.bank0 : P.bank1);
  float2 L[NS], R[NS], s[NS];
#pragma unroll
  for (int k = 0; k < NS; ++k) {
    const int c = c0 + k * CPB + cl;
    L[k] = lam[(size_t)c * M + m];
    R[k] = res[(size_t)c * M + m];
    s[k] = slot >= 0 ? cur[((size_t)slot * d + c) * M + m] : make_float2(0.f, 0.f);
  }
  const int tiles[3] = {c0 / TILE_M, (d + c0) / TILE_M, (2 * d + c0) / TILE_M};
  if (!row_wait_tiles(P, tiles, 3, ab, s_flag)) return false;
  const SrcSlots src{P.ws, P.tab, NTOK};
  for (int e = rt; e < n * CH; e += E_ROWT) {
    const int t = e / CH, cc = c0 + e % CH;
    const float a = stored<bf16>(src.get(src.at(cc), t, cc));
    const float b = stored<bf16>(src.get(src.at(d + cc), t, d + cc));
    const float v = stored<bf16>(src.get(src.at(2 * d + cc), t, 2 * d + cc));
    a_s[t * CH + e % CH] = a;
    z_s[t * CH + e % CH] = b * v;
  }
  row_sync();
  bf16* g = static_cast<bf16*>(P.out);
  for (int t = 0; t < n; ++t) {
#pragma unroll
    for (int k = 0; k < NS; ++k) {
      const int ci = k * CPB + cl, c = c0 + ci;
      const float z = z_s[t * CH + ci];
      const float sr = fmaf(L[k].x, s[k].x, fmaf(-L[k].y, s[k].y, z));
      const float si = fmaf(L[k].x, s[k].y, L[k].y * s[k].x);
      s[k] = make_float2(sr, si);
      dst[((size_t)t * d + c) * M + m] = s[k];
      float y = fmaf(R[k].x, s[k].x, -R[k].y * s[k].y);
#pragma unroll
      for (int o = M / 2; o > 0; o >>= 1) y += __shfl_xor_sync(0xffffffffu, y, o);
      if (m == 0) g[(size_t)t * d + c] = __float2bfloat16_rn(a_s[t * CH + ci] * y);
    }
  }
  row_signal(P.ready, true);
  row_sync();
  return true;
}

// Residual add of one 128-column tile from the out / down GEMM's slots and
// the tile's per-row sum of squares (resid_norm_kernel's arithmetic: lane l
// owns columns 4l .. 4l+3, the squares meet in the GEMM epilogue's order);
// then, once every tile of the rows is added, the RMSNorm of this tile: the
// row's sum of squares is its tile sums added in tile order.
__device__ bool resid_item(const EngPhase& P, int t, int n, int d, float eps, Abort ab, volatile int* s_flag) {
  if (!row_wait_tiles(P, &t, 1, ab, s_flag)) return false;
  const int rt = threadIdx.x - E_ROW0 * 32, lane = rt & 31, warp = rt >> 5;
  const SrcSlots src{P.ws, P.tab, NTOK};
  {
    const int col = t * TILE_M + 4 * lane;
    const SrcSlots::Col c = src.at(col);
    const size_t stride = (size_t)src.rows * TILE_M;
    for (int r = warp; r < n; r += E_ROWW) {
      float* xr = P.X + (size_t)r * d + col;
      const float* p = c.p + (size_t)r * TILE_M;
      float4 x = __ldcg(reinterpret_cast<const float4*>(xr));
      const float4 v0 = __ldcg(reinterpret_cast<const float4*>(p));
      float4 a[SLOTS_RESID_MAX];
#pragma unroll
      for (int q = 1; q < SLOTS_RESID_MAX; ++q)
        a[q] = c.cnt > q ? __ldcg(reinterpret_cast<const float4*>(p + q * stride)) : make_float4(0.f, 0.f, 0.f, 0.f);
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int q = 1; q < SLOTS_RESID_MAX; ++q) v.x += a[q].x, v.y += a[q].y, v.z += a[q].z, v.w += a[q].w;
      x.x += v0.x + v.x;
      x.y += v0.y + v.y;
      x.z += v0.z + v.z;
      x.w += v0.w + v.w;
      __stcg(reinterpret_cast<float4*>(xr), x);
      float q4[4] = {x.x * x.x, x.y * x.y, x.z * x.z, x.w * x.w};
#pragma unroll
      for (int o = 4; o > 0; o >>= 1)  // column xor 16, 8, 4
#pragma unroll
        for (int k = 0; k < 4; ++k) q4[k] += __shfl_xor_sync(0xffffffffu, q4[k], o);
      const float wsum = (q4[0] + q4[2]) + (q4[1] + q4[3]);  // column xor 2, then 1
      const float w1 = __shfl_sync(0xffffffffu, wsum, 8), w2 = __shfl_sync(0xffffffffu, wsum, 16);
      const float w3 = __shfl_sync(0xffffffffu, wsum, 24);
      if (lane == 0) __stcg(P.ss + (size_t)t * ROWS_MAX + r, ((wsum + w1) + w2) + w3);
    }
  }
  row_sync();
  if (rt == 0) {
    red_release_add(P.done, 1);
    *s_flag = e_count_wait(P.done, d / TILE_M, ab) ? 1 : 0;
  }
  row_sync();
  const bool ok = *s_flag != 0;
  row_sync();
  if (!ok) return false;
  const int r = rt >> 4, q = rt & 15;
  if (r < n) {
    const int ntiles = d / TILE_M;
    float tot = 0.f;
    for (int k = 0; k < ntiles; ++k) tot += __ldcg(P.ss + (size_t)k * ROWS_MAX + r);
    const float den = sqrtf(tot / (float)d + eps), rden = 1.f / den;
    const int col = t * TILE_M + 8 * q;
    const float4 x0 = __ldcg(reinterpret_cast<const float4*>(P.X + (size_t)r * d + col));
    const float4 x1 = __ldcg(reinterpret_cast<const float4*>(P.X + (size_t)r * d + col + 4));
    const float xs[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
    bf16* xo = static_cast<bf16*>(P.out) + (size_t)r * P.out_ld + col;
#pragma unroll
    for (int k = 0; k < 8; ++k) xo[k] = __float2bfloat16_rn(div_row(xs[k], den, rden));
  }
  row_signal(P.ready, true);
  return true;
}

// SiLU-and-multiply of gate/up tiles j*sub .. j*sub+sub-1 (the packed
// gate/up rows interleave 64 gate and 64 up rows per tile): tile t gives h
// columns 64t .. 64t+63 (mlp_act_kernel's arithmetic).
__device__ bool act_item(const EngPhase& P, int j, int n, Abort ab, volatile int* s_flag) {
  int tiles[2];
  int k = 0;
  for (; k < P.sub && j * P.sub + k < P.T; ++k) tiles[k] = j * P.sub + k;
  if (!row_wait_tiles(P, tiles, k, ab, s_flag)) return false;
  const int rt = threadIdx.x - E_ROW0 * 32;
  const int r = rt >> 4, q = rt & 15;
  if (r < n) {
    const SrcSlots src{P.ws, P.tab, NTOK};
    bf16* h = static_cast<bf16*>(P.out) + (size_t)r * P.out_ld;
    for (int i = 0; i < k; ++i) {
      const int t = tiles[i];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int jj = 4 * q + e;  // column within the tile's 64 outputs
        const int gj = t * TILE_M + jj, uj = gj + TILE_M / 2;
        const float gt = src.get(src.at(gj), r, gj), up = src.get(src.at(uj), r, uj);
        h[t * (TILE_M / 2) + jj] = __float2bfloat16_rn(silu_f(gt) * up);
      }
    }
  }
  row_signal(P.ready, true);
  return true;
}

// Logits of head tile t from its slots (the cluster fixup's order).
__device__ bool logits_item(const EngPhase& P, int t, int n, float* logits, int V, Abort ab, volatile int* s_flag) {
  if (!row_wait_tiles(P, &t, 1, ab, s_flag)) return false;
  const int rt = threadIdx.x - E_ROW0 * 32;
  const SrcSlots src{P.ws, P.tab, NTOK};
  const int col = t * TILE_M + (rt & (TILE_M - 1));
  const SrcSlots::Col c = src.at(col);
  for (int r = rt >> 7; r < n; r += E_ROWT / TILE_M) logits[(size_t)r * V + col] = src.get<8>(c, r, col);
  return true;
}

template <int M>
__device__ bool iir_sub(const EngPhase& P, int j, const EngArgs& a, float* sm, Abort ab, volatile int* f) {
  return P.sub == 2 ? iir_item<M, 2>(P, j, a.n, a.d, a.book, sm, ab, f) : iir_item<M, 1>(P, j, a.n, a.d, a.book, sm, ab, f);
}

__device__ bool row_item(const EngPhase& P, int j, const EngArgs& a, float* sm, Abort ab, volatile int* f) {
  switch (P.kind) {
    case ENG_FIR: {
      const int NW = min(8, P.L);
      int J = 1;
      while (J * NW < P.L) J <<= 1;
      switch (J) {
        case 1: return fir_item<1>(P, j, a.n, a.d, a.book, sm, ab, f);
        case 2: return fir_item<2>(P, j, a.n, a.d, a.book, sm, ab, f);
        case 4: return fir_item<4>(P, j, a.n, a.d, a.book, sm, ab, f);
        case 8: return fir_item<8>(P, j, a.n, a.d, a.book, sm, ab, f);
        default: return fir_item<16>(P, j, a.n, a.d, a.book, sm, ab, f);  // L <= 128 (checked on the host)
      }
    }
    case ENG_IIR:
      switch (P.L) {
        case 1: return iir_sub<1>(P, j, a, sm, ab, f);
        case 2: return iir_sub<2>(P, j, a, sm, ab, f);
        case 4: return iir_sub<4>(P, j, a, sm, ab, f);
        case 8: return iir_sub<8>(P, j, a, sm, ab, f);
        case 16: return iir_sub<16>(P, j, a, sm, ab, f);
        default: return iir_sub<32>(P, j, a, sm, ab, f);
      }
    case ENG_RESID: return resid_item(P, j, a.n, a.d, a.eps, ab, f);
    case ENG_ACT: return act_item(P, j, a.n, ab, f);
    case ENG_LOGITS: return logits_item(P, j, a.n, a.logits, a.V, ab, f);
    default: return true;
  }
}

__global__ void __launch_bounds__(E_THREADS, 1)
    engine_kernel(const __grid_constant__ CUtensorMap m_xn, const __grid_constant__ CUtensorMap m_g,
                  const __grid_constant__ CUtensorMap m_h, const __grid_constant__ EngArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t* sA = smem;
  uint8_t* sB = smem + E_S * EA_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + E_BAR_OFF);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3 * E_S + 5);
  volatile int* abort_local = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* s_ok = reinterpret_cast<volatile int*>(tmem_slot + 2);   // epilogue
  volatile int* s_row = reinterpret_cast<volatile int*>(tmem_slot + 3);  // row work
  volatile int* s_prod = reinterpret_cast<volatile int*>(tmem_slot + 4); // units the producer has issued
  float* row_sm = reinterpret_cast<float*>(smem + E_ROW_OFF);
  auto w_full = [&](int s) { return smem_u32(bars + s); };
  auto b_full = [&](int s) { return smem_u32(bars + E_S + s); };
  auto empty = [&](int s) { return smem_u32(bars + 2 * E_S + s); };
  auto acc_full = [&](int b) { return smem_u32(bars + 3 * E_S + b); };
  auto acc_empty = [&](int b) { return smem_u32(bars + 3 * E_S + 2 + b); };
  const uint32_t drain = smem_u32(bars + 3 * E_S + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x;
  const Abort ab{abort_local, a.gabort};
  const EngPhase* prog = a.prog;

  if (threadIdx.x == 0) {
    for (int s = 0; s < E_S; ++s) {
      mbar_init(w_full(s), 1);
      mbar_init(b_full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(acc_full(b), 1);
      mbar_init(acc_empty(b), 128);
    }
    mbar_init(drain, 1);
    *abort_local = 0;
    *s_prod = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&m_xn)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&m_g)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&m_h)) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(32)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ---------------- weight producer: tight loop, one bulk copy per unit
    const uint64_t pol = policy_evict_first();
    long long i = 0;
    bool stop = false;
    for (int ph = a.ph0; ph < a.ph1 && !stop; ++ph) {
      const EngPhase& P = prog[ph];
      if (P.kind != ENG_GEMM) continue;
      long long ub, ue;
      unit_range(P, c, &ub, &ue);
      if (ub >= ue) continue;
      const uint8_t* wp = P.wpk + (size_t)c * EA_BYTES;
      const size_t step = (size_t)P.G * EA_BYTES;
      for (long long u = ub; u < ue; ++u, ++i) {
        const int s = (int)(i & (E_S - 1));
        if (i >= E_S && !e_mbar_wait(empty(s), (uint32_t)((i >> E_SLOG) - 1) & 1, ab)) {
          stop = true;
          break;
        }
        mbar_expect_tx(w_full(s), EA_BYTES);
        bulk_load(smem_u32(sA + s * EA_BYTES), wp, EA_BYTES, w_full(s), pol);
        wp += step;
        *s_prod = (int)(i + 1);
      }
    }
    for (long long j = i > E_S ? i - E_S : 0; j < i; ++j)
      drain_wait(w_full((int)(j & (E_S - 1))), (uint32_t)(j >> E_SLOG) & 1);
  } else if (warp == 3 && lane == 0) {
    // ---------------- L2 prefetch: the units E_S .. E_S + E_PF - 1 beyond the
    // producer's front, so a stall of the ring does not stop the HBM stream
    long long i = 0;
    bool stop = false;
    const uint64_t t0 = gtimer();
    for (int ph = a.ph0; ph < a.ph1 && !stop; ++ph) {
      const EngPhase& P = prog[ph];
      if (P.kind != ENG_GEMM) continue;
      long long ub, ue;
      unit_range(P, c, &ub, &ue);
      if (ub >= ue) continue;
      const uint8_t* wp = P.wpk + (size_t)c * EA_BYTES;
      const size_t step = (size_t)P.G * EA_BYTES;
      for (long long u = ub; u < ue; ++u, ++i, wp += step) {
        if (i < E_S) continue;  // the ring's first fill
        while (i >= (long long)*s_prod + E_S + E_PF) {
          if (aborted(ab) || gtimer() - t0 > E_WAIT_NS) {
            stop = true;
            break;
          }
          __nanosleep(256);
        }
        if (stop) break;
        bulk_prefetch_l2(wp, EA_BYTES);
      }
    }
  } else if (warp == 2 && lane == 0) {
    // ---------------- activation loader
    const uint64_t pol = policy_evict_last();
    long long i = 0;
    bool ok = true;
    for (int ph = a.ph0; ph < a.ph1 && ok; ++ph) {
      const EngPhase& P = prog[ph];
      if (P.kind != ENG_GEMM) continue;
      long long ub, ue;
      unit_range(P, c, &ub, &ue);
      if (ub >= ue) continue;
      if (P.target > 0) {
        if (!e_count_wait(P.ready, P.target, ab)) break;
        fence_proxy_async_global();
      }
      const CUtensorMap* map = P.bmap == ENG_B_XN ? &m_xn : P.bmap == ENG_B_G ? &m_g : &m_h;
      const int KB = P.KB;
      int kb = (int)(ub % KB);
      for (long long u = ub; u < ue; ++u, ++i) {
        const int s = (int)(i & (E_S - 1));
        if (i >= E_S && !e_mbar_wait(empty(s), (uint32_t)((i >> E_SLOG) - 1) & 1, ab)) {
          ok = false;
          break;
        }
        mbar_expect_tx(b_full(s), EB_BYTES);
        tma_load_2d(smem_u32(sB + s * EB_BYTES), map, b_full(s), kb * TILE_K, 0, pol);
        if (++kb == KB) kb = 0;
      }
    }
    for (long long j = i > E_S ? i - E_S : 0; j < i; ++j)
      drain_wait(b_full((int)(j & (E_S - 1))), (uint32_t)(j >> E_SLOG) & 1);
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer
    const uint64_t ad0 = sw128_desc(smem_u32(sA)), bd0 = sw128_desc(smem_u32(sB));
    const uint32_t idesc = idesc_n(NTOK);
    long long i = 0;
    int seg = 0;
    bool ok = true;
    for (int ph = a.ph0; ph < a.ph1 && ok; ++ph) {
      const EngPhase& P = prog[ph];
      if (P.kind != ENG_GEMM) continue;
      long long ub, ue;
      unit_range(P, c, &ub, &ue);
      if (ub >= ue) continue;
      const int KB = P.KB;
      const int first_tile = (int)(ub / KB), nseg = (int)((ue - 1) / KB) - first_tile + 1;
      long long u = ub;
      for (int sg = 0; sg < nseg && ok; ++sg, ++seg) {
        const int b = seg & 1;
        const long long seg_end = min(ue, (long long)(first_tile + sg + 1) * KB);
        if (seg >= 2 && !e_mbar_wait(acc_empty(b), (uint32_t)((seg >> 1) - 1) & 1, ab)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t dt = tmem + (uint32_t)(b * NTOK);
        bool first = true;
        for (; u < seg_end; ++u, ++i) {
          const int s = (int)(i & (E_S - 1));
          const uint32_t par = (uint32_t)(i >> E_SLOG) & 1;
          if (!e_mbar_wait(w_full(s), par, ab)) {
            ok = false;
            break;
          }
          if (!e_mbar_wait(b_full(s), par, ab)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = ad0 + (uint64_t)(s * (EA_BYTES >> 4));
          const uint64_t bd = bd0 + (uint64_t)(s * (EB_BYTES >> 4));
#pragma unroll
          for (int k = 0; k < TILE_K / 16; ++k) mma_bf16(dt, ad + 2 * k, bd + 2 * k, idesc, (first && k == 0) ? 0u : 1u);
          first = false;
          mma_commit(empty(s));
        }
        if (ok) mma_commit(acc_full(b));
      }
    }
    mma_commit(drain);
    drain_wait(drain, 0);
  } else if (warp >= E_EPI0 && warp < E_EPI0 + 4) {
    // ---------------- epilogue: TMEM -> partial slot -> tile count
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const int g = threadIdx.x - E_EPI0 * 32;
    int seg = 0;
    bool go = true;
    for (int ph = a.ph0; ph < a.ph1 && go; ++ph) {
      const EngPhase& P = prog[ph];
      if (P.kind != ENG_GEMM) continue;
      long long ub, ue;
      unit_range(P, c, &ub, &ue);
      if (ub >= ue) continue;
      const int first_tile = (int)(ub / P.KB), nseg = (int)((ue - 1) / P.KB) - first_tile + 1;
      for (int sg = 0; sg < nseg; ++sg, ++seg) {
        const int b = seg & 1, tile = first_tile + sg;
        if (g == 0) *s_ok = e_mbar_wait(acc_full(b), (uint32_t)(seg >> 1) & 1, ab) ? 1 : 0;
        epi_sync();
        go = *s_ok != 0;
        epi_sync();
        if (!go) break;
        tc_fence_after();
        float v[NTOK];
        tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * NTOK), v);
        tc_fence_before();
        mbar_arrive(acc_empty(b));
        const int4 e = __ldg(P.tab + tile);
        float* dst = P.ws + (long long)(e.x + (c - e.z)) * NTOK * TILE_M + row;
#pragma unroll
        for (int t = 0; t < NTOK; ++t)
          if (t < a.n) __stcg(dst + t * TILE_M, v[t]);
        epi_sync();
        if (g == 0) {
          red_release_add(P.cnt + tile, 1);
        }
      }
    }
  } else if (warp >= E_ROW0) {
    // ---------------- row work
    for (int ph = a.ph0; ph < a.ph1; ++ph) {
      const EngPhase& P = prog[ph];
      if (P.kind == ENG_GEMM) continue;
      for (int j = c; j < P.G; j += gridDim.x)
        if (!row_item(P, j, a, row_sm, ab, s_row)) break;
      // all row warps leave the phase together and agree whether to go on
      row_sync();
      if (threadIdx.x == E_ROW0 * 32) *s_row = aborted(ab) ? 0 : 1;
      row_sync();
      const bool go = *s_row != 0;
      row_sync();
      if (!go) break;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(32) : "memory");
  }
  if (threadIdx.x == 0 && *abort_local) atomicOr(&a.book->status, EVS_DEV_TIMEOUT);
}

}  // namespace

int engine_row_floats(int kind, int param, int sub) {
  if (kind == ENG_FIR) {
    const int NW = param < 8 ? param : 8;
    return 32 * ((param - 1 + NTOK) + NTOK + param + NW * NTOK);
  }
  if (kind == ENG_IIR) return 2 * NTOK * sub * (256 / param);
  return 0;
}

size_t engine_smem(int row_floats) { return E_FIXED + sizeof(float) * (size_t)row_floats; }

cudaError_t launch_engine(const LaunchCtx& L, const CUtensorMap& m_xn, const CUtensorMap& m_g, const CUtensorMap& m_h,
                          const EngArgs& a, int grid) {
  const size_t smem = engine_smem(a.row_floats);
  if (smem > 232448 || a.n < 1 || a.n > NTOK || grid < 1) return cudaErrorInvalidValue;
  static size_t attr = 0;
  if (attr < smem) {
    cudaError_t e = cudaFuncSetAttribute(engine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr = smem;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(E_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = L.stream;
  // every CTA waits on counters other CTAs raise: the grid must be resident
  // all at once, which a cooperative launch guarantees (or refuses)
  cudaLaunchAttribute attr_c[1];
  attr_c[0].id = cudaLaunchAttributeCooperative;
  attr_c[0].val.cooperative = 1;
  cfg.attrs = attr_c;
  cfg.numAttrs = 1;
  count_launch();
  return cudaLaunchKernelEx(&cfg, engine_kernel, m_xn, m_g, m_h, a);
}

}  // namespace evs
