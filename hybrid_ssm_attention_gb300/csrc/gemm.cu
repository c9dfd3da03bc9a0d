// Skinny weight-streaming GEMM: partials of Y[tok][col] = sum_k X[tok][k] W[col][k]
// for a verify block of n <= 16 tokens against a [N][K] weight matrix.
//
// The verify step is bound by reading the weights once (the discussion
// post's reply, "Regime overlap": ~80% of a native step is the weight read).
// So the kernel is a weight stream: one persistent CTA per SM walks a
// contiguous range of 128x64 weight units (stream-K order), TMA brings each
// unit into a 128-byte-swizzled shared-memory ring, and one thread issues
// tcgen05.mma with the weight tile as A (M = 128 output columns) and the
// block's activations as B (N = 16 tokens), accumulating in TMEM.  Each tile
// segment's 128x16 fp32 accumulator is drained by four epilogue warps into a
// partial slot; the consumer of the GEMM sums the slots in CTA order.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdio>
#include <cstring>

#include "evs_internal.cuh"
#include "ptx.cuh"

namespace evs {

// at most MAX_CONTRIB CTAs per tile: the last one sums their slots
constexpr int MAX_CONTRIB = 8;

bool plan_gemm(int N, int K, int num_sms, GemmPlan* g) {
  const int T = (N + TILE_M - 1) / TILE_M;
  const long long U = (long long)T * ((K + TILE_K - 1) / TILE_K);
  if (T > 1024 || N < 1 || K < 1 || num_sms < 1) return false;
  return plan_gemm_grid(N, K, (int)std::min<long long>(std::min<long long>(num_sms, U), (long long)T * MAX_CONTRIB),
                        g);
}

bool plan_gemm_grid(int N, int K, int G, GemmPlan* g) {
  Partials& P = g->P;
  P = Partials{};
  P.N = N;
  const int T = (N + TILE_M - 1) / TILE_M;
  if (T > 1024 || N < 1 || K < 1 || G < 1) return false;
  P.nt = 1;
  P.KB = (K + TILE_K - 1) / TILE_K;
  P.U = (long long)T * P.KB;
  if (G > P.U || G > T * MAX_CONTRIB) return false;
  P.G = G;
  P.stages = 8;
  int base = 0;
  for (int t = 0; t < T; ++t) {
    const int c0 = unit_owner(P.U, P.G, (long long)t * P.KB);
    const int c1 = unit_owner(P.U, P.G, (long long)t * P.KB + P.KB - 1);
    g->tab[t] = make_int4(base, c1 - c0 + 1, c0, 0);
    base += c1 - c0 + 1;
  }
  g->slots = base;
  P.max_cnt = 0;
  for (int t = 0; t < T; ++t) P.max_cnt = std::max(P.max_cnt, g->tab[t].y);
  return true;
}

bool plan_gemm_cluster(int N, int K, int cl, GemmPlan* g) {
  Partials& P = g->P;
  P = Partials{};
  P.N = N;
  const int T = (N + TILE_M - 1) / TILE_M;
  if (T > 1024 || N < 1 || K < 1 || cl < 1 || cl > 8) return false;
  P.KB = (K + TILE_K - 1) / TILE_K;
  if (P.KB < cl) return false;
  P.U = (long long)T * P.KB;
  P.G = T * cl;
  P.cl = cl;
  P.nt = 1;
  // a CTA that owns a whole tile has the shared memory to itself: deepest ring
  P.stages = cl == 1 ? GEMM_MAX_STAGES : 8;
  for (int t = 0; t < T; ++t) g->tab[t] = make_int4(0, 0, 0, 0);
  g->slots = 0;
  return true;
}

// Tiles that would each be shared by several stream-K CTAs (few tiles for
// the SMs) reduce inside a cluster instead: the largest portable cluster
// size cl <= 8 with T * cl <= num_sms and KB >= cl; a single K-block gives
// tile mode (cl = 1).  Tile-rich shapes (more than num_sms / 2 tiles) keep
// stream-K (0): one tile per CTA there leaves SMs idle and measured slower.
int gemm_cluster_choice(int N, int K, int num_sms) {
  const int T = (N + TILE_M - 1) / TILE_M;
  const int KB = (K + TILE_K - 1) / TILE_K;
  if (2 * T > num_sms) return 0;
  int cl = 8;
  while (cl > 1 && (T * cl > num_sms || KB < cl)) cl >>= 1;
  return cl;
}

static bool encode_tmap(CUtensorMap* map, CUtensorMapDataType type, size_t esize, CUtensorMapSwizzle swz,
                       const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner, uint32_t box_outer,
                       char* err, size_t errlen) {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess || q != cudaDriverEntryPointSuccess || !p) {
      snprintf(err, errlen, "cuTensorMapEncodeTiled entry point unavailable");
      return false;
    }
    fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * esize};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(map, type, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(err, errlen, "cuTensorMapEncodeTiled failed (%d) for [%llu][%llu]", (int)r,
             (unsigned long long)outer, (unsigned long long)inner);
    return false;
  }
  return true;
}

bool encode_tmap_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                    uint32_t box_inner, uint32_t box_outer, char* err, size_t errlen) {
  return encode_tmap(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, CU_TENSOR_MAP_SWIZZLE_128B, base, inner, outer,
                     box_inner, box_outer, err, errlen);
}

bool encode_tmap_2d_f32(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                        uint32_t box_inner, uint32_t box_outer, char* err, size_t errlen) {
  return encode_tmap(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, CU_TENSOR_MAP_SWIZZLE_NONE, base, inner, outer,
                     box_inner, box_outer, err, errlen);
}

namespace {

constexpr int A_BYTES = TILE_M * TILE_K * 2;  // 16 KB weight tile
constexpr int B_BYTES = NTOK * TILE_K * 2;    // 2 KB activation tile
// warp 0 TMA, warp 1 MMA, warps 2-5 epilogue, warps 6-9 B-tile converters
constexpr int GEMM_THREADS = 320;
constexpr int N_CONV = 4;
constexpr size_t CL_SLOT = (size_t)NTOK * TILE_M * sizeof(float);  // one rank's accumulator
// fp32 source rows staged per stage for a converted (RMSNorm) B tile
__host__ __device__ constexpr int raw_bytes(int bsrc) { return bsrc == GEMM_B_NORM ? NTOK * TILE_K * 4 : 0; }
constexpr int SWG_BYTES = NTOK * (TILE_M / 2) * 4;  // gate/up exchange of the SwiGLU epilogue
// dynamic shared memory of a launch with S ring stages, cl cluster ranks and
// B source bsrc: alignment slack, ring (weights, B tiles, raw rows),
// barriers (full, empty, ready: S each; acc_full[2], acc_empty[2], drain),
// TMEM slot + flags, reduction scratch, converter row scales, SwiGLU
// exchange, cluster slots
__host__ __device__ constexpr size_t gemm_smem(int S, int cl, int bsrc, int nt = 1) {
  return 1024 + (size_t)S * (A_BYTES + nt * B_BYTES + raw_bytes(bsrc)) + (size_t)(3 * S + 5) * 8 + 16 +
         4 * NTOK * 4 + 2 * NTOK * 4 + SWG_BYTES + (size_t)(cl > 1 ? cl - 1 : 0) * CL_SLOT;
}
constexpr size_t GEMM_SMEM_MAX = 232448;

// Synchronisation of the 128 threads that drain a tile segment: the four
// epilogue warps (named barrier 1) in the tensor-core kernel, the whole CTA
// in the SIMT kernel.
template <bool NAMED>
__device__ __forceinline__ void group_sync() {
  if (NAMED)
    asm volatile("bar.sync 1, 128;" ::: "memory");
  else
    __syncthreads();
}

// Called by the 128 group threads (thread `row` holds column tile*128+row)
// after the CTA's partial slot for `tile` is written.  The contributor that
// arrives last sums the tile's slots in contributor order and writes the
// output of P.mode; it then re-arms the counter for the next launch.
__device__ __forceinline__ int atom_add_acq_rel(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// Writes the final sums v[] of column tile*128+row: GEMM_FINAL to P.fin,
// GEMM_RESID into P.X plus the tile's per-token sums of squares (butterfly
// within each warp, then the four warps in order), GEMM_SWIGLU the bf16
// activation of the tile's 64 gate / 64 up columns (exchanged through
// s_xch).  Called by the 128 group threads.
template <bool NAMED>
__device__ void tile_output(const Partials& P, int tile, int row, const float* v, float* s_red, float* s_xch,
                            const float* xpre = nullptr, int chunk = 0) {
  const int col = tile * TILE_M + row;
  const bool ok = col < P.N;
  const int r0 = chunk * NTOK;  // this chunk's first token row
  const int n = min(NTOK, P.n - r0);
  if (P.mode == GEMM_FINAL) {
    if (ok) {
#pragma unroll
      for (int t = 0; t < NTOK; ++t)
        if (t < n) P.fin[(size_t)(r0 + t) * P.fin_ld + col] = v[t];
    }
  } else if (P.mode == GEMM_SWIGLU) {
    constexpr int HALF = TILE_M / 2;
    if (row >= HALF) {
#pragma unroll
      for (int t = 0; t < NTOK; ++t)
        if (t < n) s_xch[t * HALF + row - HALF] = v[t];
    }
    group_sync<NAMED>();
    const int hc = tile * HALF + row;
    if (row < HALF && hc < P.h_cols) {
#pragma unroll
      for (int t = 0; t < NTOK; ++t)
        if (t < n)
          P.hout[(size_t)(r0 + t) * P.h_cols + hc] = __float2bfloat16_rn(silu_f(v[t]) * s_xch[t * HALF + row]);
    }
    group_sync<NAMED>();  // the exchange buffer is free again
  } else {
    const int lane = row & 31, w = row >> 5;
    // all residual loads first (independent, in flight together), then the
    // updates and the per-token butterflies
    float x[NTOK];
#pragma unroll
    for (int t = 0; t < NTOK; ++t)
      x[t] = (t < n && ok) ? (xpre ? xpre[t] : P.X[(size_t)(r0 + t) * P.N + col]) : 0.f;
#pragma unroll
    for (int t = 0; t < NTOK; ++t)
      if (t < n && ok) {
        x[t] += v[t];
        P.X[(size_t)(r0 + t) * P.N + col] = x[t];
      }
#pragma unroll
    for (int t = 0; t < NTOK; ++t) {
      float sq = x[t] * x[t];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
      if (lane == 0) s_red[w * NTOK + t] = sq;
    }
    group_sync<NAMED>();
    if (row < NTOK)
      P.ss[tile * ROWS_MAX + r0 + row] =
          ((s_red[row] + s_red[NTOK + row]) + s_red[2 * NTOK + row]) + s_red[3 * NTOK + row];
    group_sync<NAMED>();  // s_red is free again (the next chunk reuses it)
  }
}

// MC: the launch may carry several row chunks (P.nt); otherwise exactly one
template <bool NAMED, bool MC = false>
__device__ void tile_done(const Partials& P, int tile, int row, volatile int* s_flag, float* s_red, float* s_xch) {
  // The barrier orders the group's slot stores before thread 0's
  // acquire-release increment (release publishes them to the GPU; acquire
  // makes the other contributors' stores visible to whoever finishes last,
  // and the next barrier extends that to the whole group).
  group_sync<NAMED>();
  if (row == 0) *s_flag = atom_add_acq_rel(P.cnt + tile, 1);
  group_sync<NAMED>();
  const int4 e = __ldg(P.tab + tile);
  const int arrived = *s_flag;
  group_sync<NAMED>();  // every thread has read the flag before it is reused
  if (arrived != e.y - 1) return;
  const int nt = MC ? P.nt : 1;
  const size_t slot_f = (size_t)nt * NTOK * TILE_M;  // floats per slot
  for (int c = 0; c < nt; ++c) {
    const int n = min(NTOK, P.n - c * NTOK);
    const float* p = P.ws + (size_t)e.x * slot_f + (size_t)c * NTOK * TILE_M + row;
    // Fixed order: the later contributors' slots 1..count-1 in order, then
    // the first contributor's slot is added to that sum.  Slots are loaded
    // four at a time.
    float v[NTOK], v0[NTOK];
#pragma unroll
    for (int t = 0; t < NTOK; ++t) v[t] = 0.f, v0[t] = (t < n) ? __ldcg(p + t * TILE_M) : 0.f;
    for (int j0 = 1; j0 < e.y; j0 += 4) {
      float a[4][NTOK];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float* q = p + (size_t)(j0 + k) * slot_f;
#pragma unroll
        for (int t = 0; t < NTOK; ++t) a[k][t] = (j0 + k < e.y && t < n) ? __ldcg(q + t * TILE_M) : 0.f;
      }
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (j0 + k < e.y) {
#pragma unroll
          for (int t = 0; t < NTOK; ++t) v[t] += a[k][t];
        }
    }
#pragma unroll
    for (int t = 0; t < NTOK; ++t) v[t] = v0[t] + v[t];
    tile_output<NAMED>(P, tile, row, v, s_red, s_xch, nullptr, c);
  }
  if (row == 0) P.cnt[tile] = 0;
}

// At most 144 registers a thread (no spills): a 320-thread block then leaves
// a 256-thread, 72-register mixer CTA room on the SM to start its prologue
// while the GEMM drains.
// MC: several 16-row chunks (P.nt > 1); a separate instance so that the
// one-chunk kernel keeps its register allocation.  It holds the wider
// epilogue's state in 168 registers (no spills; a 72-register mixer CTA
// still fits beside it).
template <bool MC>
__global__ void __maxnreg__(MC ? 168 : 144)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap xmap,
                   const __grid_constant__ CUtensorMap nmap, Partials P, int* err_flag) {
  extern __shared__ uint8_t smem_raw[];
  const int STAGES = P.stages;  // ring depth of this launch
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const int RAW = raw_bytes(P.bsrc);
  // token rows in NT chunks of 16: MMA N = 16 NT, B stage = NT 2 KB tiles
  // (consecutive 8-row core-matrix groups, so one descriptor spans them all)
  const int NT = MC ? P.nt : 1;
  const int NN = NTOK * NT;
  const int BST = NT * B_BYTES;
  // TMEM columns: two accumulators of NN columns, a power of two >= 32
  const uint32_t tmem_cols = NN <= 16 ? 32u : NN <= 32 ? 64u : NN <= 64 ? 128u : 256u;
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  uint8_t* sR = sB + STAGES * BST;  // fp32 source rows of converted B tiles
  uint64_t* bars = reinterpret_cast<uint64_t*>(sR + STAGES * RAW);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3 * STAGES + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* s_flag = reinterpret_cast<volatile int*>(tmem_slot + 2);
  volatile int* s_ok = reinterpret_cast<volatile int*>(tmem_slot + 3);
  float* s_red = reinterpret_cast<float*>(tmem_slot + 4);  // [4][NTOK]
  float* s_scale = s_red + 4 * NTOK;  // [2][NTOK] RMSNorm divisors and their reciprocals
  float* s_xch = s_scale + 2 * NTOK;  // [NTOK][64] SwiGLU up sums
  float* s_cl = s_xch + SWG_BYTES / 4;  // cluster mode, rank 0: [cl-1][NTOK][TILE_M] partials of ranks 1..cl-1
  auto full = [&](int s) { return smem_u32(bars + s); };
  auto empty = [&](int s) { return smem_u32(bars + STAGES + s); };
  auto ready = [&](int s) { return smem_u32(bars + 2 * STAGES + s); };  // converted B tile written
  auto acc_full = [&](int b) { return smem_u32(bars + 3 * STAGES + b); };
  auto acc_empty = [&](int b) { return smem_u32(bars + 3 * STAGES + 2 + b); };
  const uint32_t drain = smem_u32(bars + 3 * STAGES + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x;
  // cl >= 1: one tile per CTA group (cl == 1: a whole tile per CTA, no
  // reduction; cl > 1: K split over the ranks of a cluster); cl == 0: stream-K
  const bool clmode = P.cl >= 1;
  int crank = 0;
  long long ub, ue;
  if (clmode) {
    if (P.cl > 1) asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(crank));
    const long long t0 = (long long)(c / P.cl) * P.KB;
    ub = t0 + (long long)crank * P.KB / P.cl;
    ue = t0 + (long long)(crank + 1) * P.KB / P.cl;
  } else {
    ub = unit_begin(P.U, P.G, c);
    ue = unit_begin(P.U, P.G, c + 1);
  }
  const long long nunits = ue - ub;
  const int first_tile = (int)(ub / P.KB);
  const int nseg = (int)((ue - 1) / P.KB) - first_tile + 1;
  float vkeep[NTOK];  // cluster mode: this CTA's accumulator column, kept across the cluster barrier
  float xpre[NTOK];   // cluster rank 0, residual mode: the tile's residual rows, loaded early
  bool have_x = false;
#pragma unroll
  for (int t = 0; t < NTOK; ++t) vkeep[t] = 0.f, xpre[t] = 0.f;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
      mbar_init(ready(s), N_CONV);  // one arrival per converter warp
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(acc_full(b), 1);
      mbar_init(acc_empty(b), 128);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    if (!P.wpk) asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&wmap)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&xmap)) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(tmem_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_trigger();

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer
    const uint64_t pol_w = policy_evict_first(), pol_x = policy_evict_last();
    const int pre = (int)std::min<long long>(STAGES, nunits);
    // weight tiles do not depend on the preceding kernel: start streaming now
    // Unit cursor (K-block kb of tile t; packed block wp) advanced
    // incrementally: this thread's per-unit work is on the critical path.
    const int KB = P.KB;
    const int kb0 = (int)(ub % KB), t0 = (int)(ub / KB);
    const uint8_t* wp0 = P.wpk ? P.wpk + (size_t)c * A_BYTES : nullptr;
    const size_t wstep = (size_t)P.G * A_BYTES;
    const uint32_t sA_u = smem_u32(sA), sB_u = smem_u32(sB), sR_u = smem_u32(sR), full0 = full(0);
    auto load_w = [&](int s, int kb, int t, const uint8_t* wp) {
      if (wp)
        bulk_load(sA_u + s * A_BYTES, wp, A_BYTES, full0 + 8 * s, pol_w);
      else
        tma_load_2d(sA_u + s * A_BYTES, &wmap, full0 + 8 * s, kb * TILE_K, t * TILE_M, pol_w);
    };
    // activations: the bf16 B tile itself, or the fp32 rows it is built from
    auto load_b = [&](int s, int kb) {
      const int x = kb * TILE_K;
      if (P.bsrc == GEMM_B_TMA) {
        for (int ch = 0; ch < NT; ++ch)
          tma_load_2d(sB_u + s * BST + ch * B_BYTES, &xmap, full0 + 8 * s, x, ch * NTOK, pol_x);
      } else {
        tma_load_2d(sR_u + s * RAW, &xmap, full0 + 8 * s, x, 0, pol_x);
      }
    };
    const uint32_t stage_tx = A_BYTES + (P.bsrc == GEMM_B_TMA ? BST : RAW);
    int kb = kb0, t = t0;
    const uint8_t* wp = wp0;
    for (int i = 0; i < pre; ++i) {
      mbar_expect_tx(full0 + 8 * i, stage_tx);
      load_w(i, kb, t, wp);
      if (++kb == KB) kb = 0, ++t;
      if (wp) wp += wstep;
    }
    pdl_wait();  // activations are written by the preceding kernel
    for (int i = 0, k2 = kb0; i < pre; ++i) {
      load_b(i, k2);
      if (++k2 == KB) k2 = 0;
    }
    // refills: unit i >= STAGES reuses stage i % STAGES once the MMA of unit
    // i - STAGES released it (empty phase (i / STAGES - 1) & 1)
    const uint32_t empty0 = empty(0);
    int s = 0;
    uint32_t ph = 0;
    long long i = pre;
    for (; i < nunits; ++i) {
      if (!mbar_wait(empty0 + 8 * s, ph, abort_flag)) break;
      mbar_expect_tx(full0 + 8 * s, stage_tx);
      load_w(s, kb, t, wp);
      load_b(s, kb);
      if (++kb == KB) kb = 0, ++t;
      if (wp) wp += wstep;
      if (++s == STAGES) s = 0, ph ^= 1;
    }
    // All own tiles are requested: keep HBM busy through this kernel's tail
    // and the consumers that follow by pulling the first units of the next
    // weight matrix (the ones the CTA of the same index will read first)
    // into L2.
    if (i == nunits && P.pf_units > 0 && c < P.nG) {
      long long nb, ne;
      if (P.ncl >= 1) {
        const long long t0 = (long long)(c / P.ncl) * P.nKB;
        nb = t0 + (long long)(c % P.ncl) * P.nKB / P.ncl;
        ne = t0 + (long long)(c % P.ncl + 1) * P.nKB / P.ncl;
      } else {
        nb = unit_begin(P.nU, P.nG, c);
        ne = unit_begin(P.nU, P.nG, c + 1);
      }
      const long long stop = std::min<long long>(ne, nb + P.pf_units);
      if (P.nwpk) {
        for (long long u = nb; u < stop; ++u) bulk_prefetch_l2(P.nwpk + ((u - nb) * P.nG + c) * A_BYTES, A_BYTES);
      } else {
        for (long long u = nb; u < stop; ++u)
          tma_prefetch_l2(&nmap, (int)(u % P.nKB) * TILE_K, (int)(u / P.nKB) * TILE_M);
      }
    }
    // make sure no copy into this CTA's shared memory is still in flight
    for (long long j = std::max<long long>(0, i - STAGES); j < i; ++j) {
      volatile int local_abort = 0;
      mbar_wait(full((int)(j % STAGES)), (uint32_t)(j / STAGES) & 1, &local_abort);
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer
    long long i = 0;
    bool ok = true;
    // stage / phase cursor and descriptors advanced incrementally (the
    // descriptors' 14-bit start-address field holds any shared address)
    const uint32_t wait0 = P.bsrc == GEMM_B_TMA ? full(0) : ready(0), empty0 = empty(0);
    const uint64_t ad0 = sw128_desc(smem_u32(sA)), bd0 = sw128_desc(smem_u32(sB));
    const uint32_t idesc = idesc_n(NN);
    int s = 0;
    uint32_t ph = 0;
    for (int seg = 0; seg < nseg && ok; ++seg) {
      const int tile = first_tile + seg;
      const long long seg_end = std::min<long long>(ue, (long long)(tile + 1) * P.KB);
      const int b = seg & 1;
      if (seg >= 2 && !mbar_wait(acc_empty(b), (uint32_t)((seg >> 1) - 1) & 1, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t dt = tmem + (uint32_t)(b * NN);
      bool first = true;
      const int cnt = (int)(seg_end - (ub + i));
      for (int j = 0; j < cnt; ++j, ++i) {
        if (!mbar_wait(wait0 + 8 * s, ph, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t ad = ad0 + (uint64_t)(s * (A_BYTES >> 4));
        const uint64_t bd = bd0 + (uint64_t)(s * (BST >> 4));
#pragma unroll
        for (int k = 0; k < TILE_K / 16; ++k)  // 16 bf16 = 32 bytes per MMA step along K
          mma_bf16(dt, ad + 2 * k, bd + 2 * k, idesc, (first && k == 0) ? 0u : 1u);
        first = false;
        mma_commit(empty0 + 8 * s);
        if (++s == STAGES) s = 0, ph ^= 1;
      }
      if (ok) mma_commit(acc_full(b));
    }
    // wait for every issued MMA before TMEM is released
    mma_commit(drain);
    volatile int local_abort = 0;
    mbar_wait(drain, 0, &local_abort);
  } else if (warp >= 2 && warp < 6) {
    // ---------------- epilogue: TMEM -> partial slots -> tile fixup
    const int q = warp & 3;         // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;  // column within the tile
    const int g = threadIdx.x - 64; // index within the epilogue group
    // cluster rank 0 of a residual GEMM: the residual rows of its tile do not
    // depend on this GEMM; fetch them while the weights stream
    if (clmode && crank == 0 && P.mode == GEMM_RESID) {
      pdl_wait();
      const int col = first_tile * TILE_M + row;
#pragma unroll
      for (int t = 0; t < NTOK; ++t) xpre[t] = (t < P.n && col < P.N) ? __ldcg(P.X + (size_t)t * P.N + col) : 0.f;
      have_x = true;
    }
    for (int seg = 0; seg < nseg; ++seg) {
      const int b = seg & 1;
      const int tile = first_tile + seg;
      // one thread waits; the decision is shared so the group stays in step
      if (g == 0) *s_ok = mbar_wait(acc_full(b), (uint32_t)(seg >> 1) & 1, abort_flag) ? 1 : 0;
      group_sync<true>();
      const int go = *s_ok;
      group_sync<true>();
      if (!go) break;
      tc_fence_after();
      const uint32_t tacc = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * NN);
      float v[NTOK];
      tmem_ld16(tacc, v);
      if (NT == 1) {
        tc_fence_before();
        mbar_arrive(acc_empty(b));
      }
      if (clmode) {
        // ranks 1..cl-1 send their column to rank 0's shared memory
        if (crank == 0) {
#pragma unroll
          for (int j = 0; j < NTOK; ++j) vkeep[j] = v[j];
        } else {
          const uint32_t local = smem_u32(s_cl + ((size_t)(crank - 1) * NTOK) * TILE_M + row);
          uint32_t remote;
          asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(0));
#pragma unroll
          for (int j = 0; j < NTOK; ++j)
            if (j < P.n)
              asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote + (uint32_t)(j * TILE_M * 4)), "f"(v[j])
                           : "memory");
        }
        continue;
      }
      const int4 e = __ldg(P.tab + tile);
      const long long slot = e.x + (c - e.z);
      float* dst = P.ws + slot * NN * TILE_M + row;
      // row chunk by row chunk into the slot ([NT][16][128]); with several
      // chunks the accumulator is released after the last one leaves TMEM
      for (int ch = 0;;) {
        const int nc = P.n - ch * NTOK;
#pragma unroll
        for (int j = 0; j < NTOK; ++j)
          if (j < nc) __stcg(dst + j * TILE_M, v[j]);
        if (++ch == NT) break;
        tmem_ld16(tacc + (uint32_t)(ch * NTOK), v);
        dst += NTOK * TILE_M;
      }
      if (NT > 1) {
        tc_fence_before();
        mbar_arrive(acc_empty(b));
      }
      if (P.mode != GEMM_SLOTS) tile_done<true, MC>(P, tile, row, s_flag, s_red, s_xch);
    }
  } else if (warp >= 6 && P.bsrc != GEMM_B_TMA) {
    // ---------------- B-tile converters: fp32 residual rows (staged by TMA)
    // -> bf16 RMSNorm rows in the 128-byte swizzled K-major layout the MMA
    // reads.  Every unit is shared by the N_CONV warps (warp w: rows
    // 4w .. 4w+3), so the first tile is ready after a quarter of the work.
    const int w = warp - 6;
    pdl_wait();  // ss_in and X are written by the preceding kernels
    if (w == 0 && lane < NTOK) {
      // row divisor sqrt(mean square + eps): per-tile sums added in tile
      // order, loaded sixteen at a time
      const float* p = P.ss_in + lane;
      float tot = 0.f;
      int k = 0;
      for (; k + 16 <= P.ss_tiles; k += 16) {
        float a[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) a[e] = __ldcg(p + (k + e) * ROWS_MAX);
#pragma unroll
        for (int e = 0; e < 16; ++e) tot += a[e];
      }
      for (; k < P.ss_tiles; ++k) tot += __ldcg(p + k * ROWS_MAX);
      const float den = sqrtf(tot / (float)P.norm_d + P.eps);
      s_scale[lane] = den;
      s_scale[NTOK + lane] = 1.f / den;
    }
    asm volatile("bar.sync 2, %0;" ::"n"(N_CONV * 32) : "memory");
    // lane -> (row parity, float4 column group): one instruction covers two
    // whole 256-byte source rows and two 128-byte B rows (no bank conflicts)
    const int cq = lane & 15, rh = lane >> 4;
    const int r0 = 4 * w + rh, r1 = r0 + 2;  // this lane's two rows
    const float den0 = s_scale[r0], rd0 = s_scale[NTOK + r0];
    const float den1 = s_scale[r1], rd1 = s_scale[NTOK + r1];
    int s = 0, kb = (int)(ub % P.KB);
    uint32_t ph = 0;
    for (long long i = 0; i < nunits; ++i) {
      if (!warp_wait(full(s), ph, abort_flag)) break;
      const int col = kb * TILE_K + 4 * cq;  // first of this lane's four columns
      const float* raw = reinterpret_cast<const float*>(sR + s * RAW) + 4 * cq;
      uint8_t* dstB = sB + s * B_BYTES + (cq & 1) * 8;
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        const int r = m ? r1 : r0;
        const float den = m ? den1 : den0, rden = m ? rd1 : rd0;
        const float4 x4 = *reinterpret_cast<const float4*>(raw + r * TILE_K);
        const float v[4] = {div_row(x4.x, den, rden), div_row(x4.y, den, rden), div_row(x4.z, den, rden),
                            div_row(x4.w, den, rden)};
        uint32_t wd[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const bool lo_ok = r < P.n && col + 2 * e < P.Kdim;
          const bool hi_ok = r < P.n && col + 2 * e + 1 < P.Kdim;
          const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(lo_ok ? v[2 * e] : 0.f));
          const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(hi_ok ? v[2 * e + 1] : 0.f));
          wd[e] = lo | (hi << 16);
        }
        // 16-byte chunk j = cq / 2 of row r sits at position j ^ (r & 7)
        *reinterpret_cast<uint2*>(dstB + r * 128 + (((cq >> 1) ^ (r & 7)) << 4)) = make_uint2(wd[0], wd[1]);
      }
      // generic-proxy writes -> visible to the tensor core's async proxy
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(ready(s));
      if (++s == STAGES) s = 0, ph ^= 1;
      if (++kb == P.KB) kb = 0;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (clmode) {
    if (P.cl > 1) {
      // every thread of every rank: the partials sent to rank 0 are visible
      // after this barrier (release / acquire at cluster scope)
      asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
      asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
    }
    if (crank == 0 && warp >= 2 && warp < 6 && !*abort_flag) {
      const int row = (warp & 3) * 32 + lane;
      // the stream-K fixup's order: ranks 1..cl-1 summed in rank order, then
      // rank 0's column added (a pass planned either way rounds alike)
      if (P.cl > 1) {
        float acc[NTOK];
#pragma unroll
        for (int j = 0; j < NTOK; ++j) acc[j] = 0.f;
        for (int r = 1; r < P.cl; ++r) {
          const float* src = s_cl + ((size_t)(r - 1) * NTOK) * TILE_M + row;
#pragma unroll
          for (int j = 0; j < NTOK; ++j)
            if (j < P.n) acc[j] += src[j * TILE_M];
        }
#pragma unroll
        for (int j = 0; j < NTOK; ++j) vkeep[j] = vkeep[j] + acc[j];
      }
      tile_output<true>(P, first_tile, row, vkeep, s_red, s_xch, have_x ? xpre : nullptr);
    }
  }
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(tmem_cols) : "memory");
  }
  if (threadIdx.x == 0 && *abort_flag) atomicOr(err_flag, EVS_DEV_TIMEOUT);
}

// SIMT variant with the same unit schedule and partial layout (float32
// storage, or shapes the tensor-core path does not take).
template <typename T>
__global__ void __launch_bounds__(128) gemm_simt_kernel(const T* W, const T* X, int ldx, Partials P, int K) {
  __shared__ float xs[NTOK][TILE_K];
  __shared__ int s_flag;
  __shared__ float s_red[4 * NTOK];
  const int n = P.n;
  pdl_trigger();
  pdl_wait();
  const int c = blockIdx.x;
  const long long ub = unit_begin(P.U, P.G, c), ue = unit_begin(P.U, P.G, c + 1);
  long long u = ub;
  while (u < ue) {
    const int tile = (int)(u / P.KB);
    const long long seg_end = std::min<long long>(ue, (long long)(tile + 1) * P.KB);
    const int row = tile * TILE_M + threadIdx.x;
    float acc[NTOK];
#pragma unroll
    for (int t = 0; t < NTOK; ++t) acc[t] = 0.f;
    for (; u < seg_end; ++u) {
      const int k0 = (int)(u % P.KB) * TILE_K;
      const int kn = min(TILE_K, K - k0);
      __syncthreads();
      for (int e = threadIdx.x; e < NTOK * TILE_K; e += blockDim.x) {
        const int t = e / TILE_K, k = e % TILE_K;
        xs[t][k] = (t < n && k < kn) ? to_f(X[(size_t)t * ldx + k0 + k]) : 0.f;
      }
      __syncthreads();
      if (row < P.N) {
        const T* wr = W + (size_t)row * K + k0;
        for (int k = 0; k < kn; ++k) {
          const float w = to_f(wr[k]);
#pragma unroll
          for (int t = 0; t < NTOK; ++t) acc[t] = fmaf(w, xs[t][k], acc[t]);
        }
      }
    }
    const int4 e = __ldg(P.tab + tile);
    const long long slot = e.x + (c - e.z);
    float* dst = P.ws + slot * NTOK * TILE_M + threadIdx.x;
#pragma unroll
    for (int t = 0; t < NTOK; ++t)
      if (t < n) __stcg(dst + t * TILE_M, acc[t]);
    tile_done<false>(P, tile, threadIdx.x, &s_flag, s_red, nullptr);
  }
}

// Exercises the pipeline's bounded wait: an mbarrier that nothing ever
// arrives on, waited on with a short limit; the expiry must come back as
// EVS_DEV_TIMEOUT in *status, with the kernel returning normally.
__global__ void wait_selftest_kernel(int* status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  abort_flag = 0;
  mbar_init(smem_u32(&bar), 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  volatile int* ab = &abort_flag;
  if (!mbar_try(smem_u32(&bar), 0) && !mbar_wait_slow(smem_u32(&bar), 0, ab, limit_ns))
    atomicOr(status, EVS_DEV_TIMEOUT);
}

// One CTA per 16 KB unit u (tile-major): 128 rows x 8 chunks of 16 bytes,
// chunk j of row r stored at position j ^ (r & 7); out-of-range rows /
// columns are zero.  The block goes to i * G + c for the CTA c that owns u
// (stream-K range or cluster rank) and u's index i within that CTA.
__global__ void __launch_bounds__(256) pack_weights_kernel(const bf16* W, int N, int K, Partials P, int swg_half,
                                                           uint8_t* dst) {
  const long long u = blockIdx.x;
  const int KB = P.KB;
  const int t = (int)(u / KB), kb = (int)(u % KB);
  long long pos;
  if (P.cl >= 1) {
    const int r = (int)unit_owner(KB, P.cl, kb);
    pos = (long long)(kb - (int)unit_begin(KB, P.cl, r)) * P.G + (long long)t * P.cl + r;
  } else {
    const int c = unit_owner(P.U, P.G, u);
    pos = (u - unit_begin(P.U, P.G, c)) * P.G + c;
  }
  uint8_t* blk = dst + pos * A_BYTES;
  for (int e = threadIdx.x; e < TILE_M * 8; e += blockDim.x) {
    const int r = e >> 3, jp = e & 7, j = jp ^ (r & 7);
    constexpr int HALF = TILE_M / 2;
    const long long row = swg_half > 0 ? (r < HALF ? (long long)t * HALF + r : swg_half + (long long)t * HALF + r - HALF)
                                       : (long long)t * TILE_M + r;
    const int col = kb * TILE_K + j * 8;
    union {
      uint4 v;
      bf16 h[8];
    } x;
#pragma unroll
    for (int i = 0; i < 8; ++i)
      x.h[i] = (row < N && col + i < K) ? W[row * K + col + i] : __float2bfloat16_rn(0.f);
    *reinterpret_cast<uint4*>(blk + r * 128 + jp * 16) = x.v;
  }
}

}  // namespace

cudaError_t launch_wait_selftest(cudaStream_t stream, int* status, unsigned long long limit_ns) {
  count_launch();
  wait_selftest_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
  return cudaGetLastError();
}

int gemm_stages_for(int cl, int bsrc, int nt) {
  int S = GEMM_MAX_STAGES;
  while (S > 2 && gemm_smem(S, cl, bsrc, nt) > GEMM_SMEM_MAX) --S;
  return S;
}

cudaError_t launch_pack_weights(cudaStream_t stream, const bf16* W, int N, int K, const Partials& P, int swg_half,
                                uint8_t* dst) {
  const long long U = (long long)((N + TILE_M - 1) / TILE_M) * ((K + TILE_K - 1) / TILE_K);
  if (U < 1 || U > 0x7fffffffLL || U != P.U) return cudaErrorInvalidValue;
  if (swg_half > 0 && (N != 2 * swg_half || swg_half % (TILE_M / 2) != 0)) return cudaErrorInvalidValue;
  cudaError_t e = cudaMemsetAsync(dst, 0, packed_bytes(P), stream);  // holes
  if (e != cudaSuccess) return e;
  count_launch();
  pack_weights_kernel<<<(unsigned)U, 256, 0, stream>>>(W, N, K, P, swg_half, dst);
  return cudaGetLastError();
}

cudaError_t launch_gemm_tc(const LaunchCtx& L, const CUtensorMap& wmap, const CUtensorMap& xmap,
                           const CUtensorMap& nmap, const Partials& P, int K, int* err_flag) {
  (void)K;
  const int cl = P.cl > 1 ? P.cl : 1;
  if (P.nt < 1 || P.nt > NT_MAX || P.n < 1 || P.n > NTOK * P.nt) return cudaErrorInvalidValue;
  // several row chunks: stream-K with TMA activations only
  if (P.nt > 1 && (P.cl != 0 || P.bsrc != GEMM_B_TMA)) return cudaErrorInvalidValue;
  const size_t smem = gemm_smem(P.stages, cl, P.bsrc, P.nt);
  if (P.stages < 2 || P.stages > GEMM_MAX_STAGES || smem > GEMM_SMEM_MAX) return cudaErrorInvalidValue;
  if (P.mode == GEMM_SWIGLU && (P.N != 2 * P.h_cols || P.h_cols % (TILE_M / 2) != 0 || !P.hout))
    return cudaErrorInvalidValue;
  if (P.mode == GEMM_SLOTS && P.cl != 0) return cudaErrorInvalidValue;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e =
        cudaFuncSetAttribute(gemm_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)GEMM_SMEM_MAX);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gemm_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)GEMM_SMEM_MAX);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  // converter warps only where the B tile is built in shared memory: the
  // smaller block leaves registers for the next kernel's CTAs to start early
  const int threads = P.bsrc == GEMM_B_TMA ? GEMM_THREADS - N_CONV * 32 : GEMM_THREADS;
  if (P.nt > 1)
    return launch_cl(L, cl, gemm_tc_kernel<true>, dim3(P.G), dim3(threads), smem, wmap, xmap, nmap, P, err_flag);
  return launch_cl(L, cl, gemm_tc_kernel<false>, dim3(P.G), dim3(threads), smem, wmap, xmap, nmap, P, err_flag);
}

cudaError_t launch_gemm_simt(const LaunchCtx& L, int dtype, const void* W, const void* X, int ldx,
                             const Partials& P, int K) {
  if (P.nt != 1 || P.n < 1 || P.n > NTOK) return cudaErrorInvalidValue;
  if (dtype == EVS_BF16)
    return launch(L, gemm_simt_kernel<bf16>, dim3(P.G), dim3(128), 0, (const bf16*)W, (const bf16*)X,
                  ldx, P, K);
  return launch(L, gemm_simt_kernel<float>, dim3(P.G), dim3(128), 0, (const float*)W, (const float*)X,
                ldx, P, K);
}

}  // namespace evs
