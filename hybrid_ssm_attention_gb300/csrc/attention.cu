// Attention mixer of one verify block on bf16 caches: rotary embedding,
// append of the block's keys and values, and split-KV block-causal attention
// in one persistent kernel (EvSpark discussion post, "What we implemented":
// an attention layer appends the block's n keys and values to its cache and
// each query attends to the committed keys and the block's keys up to its
// own position; commit keeps the first keep appended rows by moving pos).
//
// Work unit = (sequence, head, split).  Split s of a head owns keys
// [s*span, (s+1)*span) with span fixed per cache, so the partition of a
// query's keys, and with it every rounding, never depends on the block size.
// One CTA per SM takes a contiguous range of the active units (their number
// follows from the committed lengths, read on the device) and runs first the
// units whose keys are all committed, then those holding the block's keys.
//
// Roles of a CTA (MW math warps + 2):
//  * warp 8 streams K and V through a ring of 64-key stages (128 KB), each
//    stage two tensor-map loads per 64 dimensions (128-byte swizzle), one
//    mbarrier pair per stage, without draining between units.  Committed
//    keys do not depend on the preceding kernel (the first kernel of a
//    verify waits for all earlier work), so streaming starts at once;
//    stages holding the block's keys wait until this CTA appended them.
//  * warps 0-7 rotate and append the block's keys / values that fall in
//    this CTA's units (a proxy fence orders the stores before the
//    tensor-map loads), then per unit rotate the head's queries.  Warps 0-3
//    take the even stages of a unit and warps 4-7 the odd ones, 16 keys per
//    warp:
//      S = Q K^T (mma.sync m16n8k16, bf16), mask, online softmax in fp32
//      in base 2, O += P V (P rounded to bf16 as the A operand, V by
//      ldmatrix.trans);
//    at the unit's end they deposit their (max, sum, O) in shared memory and
//    go on with the next unit.
//  * a merge warp folds each deposit in warp order into the split's partial
//    (max, sum of exp, unnormalised output) while the math warps stream, and
//    counts it in the head's arrival counter (the CTA's last unit, with no
//    stream left to overlap, is merged and counted by the math warps
//    themselves, eight warps instead of one); the CTA that brings the count
//    to the head's number of splits folds the partials, after its last unit,
//    in ascending split order into the mixer output and resets the counter
//    (no CTA waits for another).
// Rows of a stage past the split's end are masked (K) or zeroed in shared
// memory by the warp that owns them (V), so P = 0 never meets a non-finite
// value.  Every mbarrier wait is bounded; on expiry the CTA raises
// EVS_DEV_TIMEOUT in the pass's books, lets its copies land and returns.
#include <algorithm>

#include "ptx.cuh"

namespace evs {
namespace {

constexpr int AK_GROUP_WARPS = 4;  // math warps of a group (16 keys of a stage each)
constexpr int AK_STAGE = 64;  // keys per ring stage
constexpr int AK_BOX = 64;    // elements of one 128-byte swizzled box row

// Two configurations: for long caches MW = 8 math warps (two groups taking
// alternate stages, a 128 KB ring, one CTA per SM), fused with the rotary
// embedding, the append and the combine (FUSED): each CTA streams many
// stages.  For short caches MW = 4 (one group, a 64 KB ring, two CTAs per
// SM), between a rotary / append kernel and the combine kernel: a few stages
// per unit, all units at once, and the three launches overlap under
// dependent launch where one fused kernel would run its steps in series.
template <int DH, int MW>
struct AkLayout {
  static constexpr int MATH_THREADS = MW * 32;
  // long caches (MW = 8): a merge warp folds each unit's warp states while
  // the math warps stream the next unit; short caches (a unit or two per
  // CTA, the merge on the critical path): the math warps merge themselves
  static constexpr bool MERGE_WARP = MW == 8;
  static constexpr int THREADS = MATH_THREADS + (MERGE_WARP ? 64 : 32);  // + producer (+ merge) warp
  static constexpr int GROUPS = MW / AK_GROUP_WARPS;
  static constexpr int HALVES = DH / AK_BOX;               // boxes per key row
  static constexpr uint32_t BOX_B = AK_STAGE * 128;        // one box: 64 rows x 128 bytes
  static constexpr uint32_t TILE_B = HALVES * BOX_B;       // K (or V) of one stage
  static constexpr int NST = (MW == 8 ? 8 : 4) / HALVES;   // ring depth: 128 / 64 KB of K and V
  static constexpr uint32_t RING_B = NST * 2 * TILE_B;
  static constexpr int QP = DH + 8;                        // row pitch (floats) of q / O rows:
                                                           // 8-byte accesses of a warp hit all banks
  // rotated queries [16][QP]; warp max / sum / weight [MW][16]; warp outputs [MW][16][QP]
  static constexpr uint32_t Q_B = 16 * QP * 4;
  static constexpr uint32_t ML_B = 3 * MW * 16 * 4;
  static constexpr uint32_t OW_B = MW * 16 * QP * 4;
  static constexpr uint32_t BAR_B = (2 * NST + 1) * 8;
  // then the fold list (host-sized: at most one entry per unit of a CTA)
  static constexpr uint32_t FOLD_OFF = RING_B + Q_B + ML_B + OW_B + BAR_B + 16;
  static constexpr size_t SMEM = 1024 + FOLD_OFF;  // without the fold list
};

template <int NTHR>
__device__ __forceinline__ void math_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(NTHR) : "memory");
}
// Hand-offs between the math warps and the merge warp (NTHR = both): id 2
// "the merge area is free", id 3 "a unit's state is deposited", id 4 "every
// unit is merged and counted"; one side arrives, the other waits.
template <int ID, int NTHR>
__device__ __forceinline__ void hand_wait() {
  asm volatile("bar.sync %0, %1;" ::"n"(ID), "n"(NTHR) : "memory");
}
template <int ID, int NTHR>
__device__ __forceinline__ void hand_arrive() {
  asm volatile("bar.arrive %0, %1;" ::"n"(ID), "n"(NTHR) : "memory");
}
// Four output dims of query row t merged over the MW warp states in warp
// order (O = sum_v w_v O_v, one fused multiply-add per warp and dim, as a
// scalar loop would) and stored as one float4.
template <int MW, int QP>
__device__ __forceinline__ void merge_dims(const float* ow, const float* fw, int t, int dd, float* dst) {
  float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int v = 0; v < MW; ++v) {
    const float4 a = *reinterpret_cast<const float4*>(ow + ((size_t)v * 16 + t) * QP + dd);
    const float w = fw[v * 16 + t];
    O.x = fmaf(a.x, w, O.x);
    O.y = fmaf(a.y, w, O.y);
    O.z = fmaf(a.z, w, O.z);
    O.w = fmaf(a.w, w, O.w);
  }
  *reinterpret_cast<float4*>(dst) = O;
}
// o / l rounded to bf16, four dims stored as one 8-byte word
__device__ __forceinline__ void store_out4(bf16* dst, float4 o, float l) {
  __nv_bfloat162 lo = __floats2bfloat162_rn(o.x / l, o.y / l), hi = __floats2bfloat162_rn(o.z / l, o.w / l);
  uint2 pk;
  pk.x = *reinterpret_cast<uint32_t*>(&lo);
  pk.y = *reinterpret_cast<uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(dst) = pk;
}
// math_sync that also returns whether v held on any math thread (the same
// answer on all of them, so branches on it stay uniform)
template <int NTHR>
__device__ __forceinline__ bool math_any(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}\n"
      : "=r"(r)
      : "r"((uint32_t)v), "n"(NTHR)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const uint32_t a = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
  const uint32_t b = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
  return a | (b << 16);
}
__device__ __forceinline__ void mma16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm4(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm4_t(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
// byte offset of 16-byte chunk c of key row r in a stage tile (TMA's
// 128-byte swizzle: within each box, chunk c & 7 of row r sits at
// (c & 7) ^ (r & 7))
__device__ __forceinline__ uint32_t tile_off(int r, int c, uint32_t box_b) {
  return (uint32_t)(c >> 3) * box_b + (uint32_t)r * 128u + ((uint32_t)((c & 7) ^ (r & 7)) << 4);
}
// Bounded mbarrier wait without a call (the math warps' stage loop keeps
// its registers): false once the wait exceeded WAIT_NS or another role
// raised the abort flag.
__device__ __forceinline__ bool wait_inl(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try(bar, parity)) return true;
  const uint64_t t0 = gtimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try(bar, parity)) return true;
    if ((i & 63) == 0 && (*abort_flag || gtimer() - t0 > WAIT_NS)) {
      *abort_flag = 1;
      return false;
    }
  }
}

// Row work of NTHR cooperating threads: thread ctid owns rotation pair
// i = ctid % (DH/2) and rows ctid / (DH/2) + k * RPP; every load of a call is
// issued before any use (one round trip), rows past the block re-read its
// last row.
template <int DH, int NTHR>
struct AkRows {
  static constexpr int HALF = DH / 2;
  static constexpr int RPP = NTHR / HALF;          // rows per pass
  static constexpr int K = (16 + RPP - 1) / RPP;   // passes to cover 16 rows
};

// The block's keys / values of head h at rows t in [t0, t1): keys rotated,
// both rounded to bf16 and stored at positions pos + t.
template <typename Src, int DH, int NTHR>
__device__ __forceinline__ void append_rows(const Src& src, int d, int h, int r0, long long pos, int t0, int t1,
                                            long long ctx_max, uint64_t fx, bf16* kc, bf16* vc, int ctid) {
  using R = AkRows<DH, NTHR>;
  constexpr int HALF = R::HALF;
  const int i = ctid % HALF, tb = t0 + ctid / HALF;  // fx: the angle step of dimension pair i
  const int col = h * DH + i;
  const auto ck1 = src.at(d + col), ck2 = src.at(d + col + HALF);
  const auto cv1 = src.at(2 * d + col), cv2 = src.at(2 * d + col + HALF);
  // at most four rows of each stream in flight per thread
  constexpr int KC = R::K < 4 ? R::K : 4;
  for (int kb = 0; kb < R::K; kb += KC) {
    float k1[KC], k2[KC], v1[KC], v2[KC];
#pragma unroll
    for (int k = 0; k < KC; ++k) {
      const int t = min(tb + (kb + k) * R::RPP, t1 - 1);
      k1[k] = src.get(ck1, r0 + t, d + col);
      k2[k] = src.get(ck2, r0 + t, d + col + HALF);
      v1[k] = src.get(cv1, r0 + t, 2 * d + col);
      v2[k] = src.get(cv2, r0 + t, 2 * d + col + HALF);
    }
#pragma unroll
    for (int k = 0; k < KC; ++k) {
      const int t = tb + (kb + k) * R::RPP;
      if (t >= t1) continue;
      const float2 c = rope_cs(pos + t, fx);
      const float x1 = stored<bf16>(k1[k]), x2 = stored<bf16>(k2[k]);
      const size_t row = ((size_t)h * ctx_max + pos + t) * DH;
      kc[row + i] = __float2bfloat16_rn(rot_lo(x1, x2, c));
      kc[row + i + HALF] = __float2bfloat16_rn(rot_hi(x1, x2, c));
      vc[row + i] = __float2bfloat16_rn(v1[k]);
      vc[row + i + HALF] = __float2bfloat16_rn(v2[k]);
    }
  }
}

// Rotated queries of head h into q [16][QP] (rows past n zero), in two steps so that the loads can overlap other work: load() issues
// them, finish() rotates, rounds and stores.
template <typename Src, int DH, int QP, int NTHR>
struct QueryRows {
  using R = AkRows<DH, NTHR>;
  float q1[R::K], q2[R::K];
  __device__ __forceinline__ void load(const Src& src, int h, int r0, int n, int ctid) {
    const int i = ctid % R::HALF, tb = ctid / R::HALF, col = h * DH + i;
    const auto ca = src.at(col), cb = src.at(col + R::HALF);
#pragma unroll
    for (int k = 0; k < R::K; ++k) {
      const int t = min(tb + k * R::RPP, n - 1);
      q1[k] = src.get(ca, r0 + t, col);
      q2[k] = src.get(cb, r0 + t, col + R::HALF);
    }
  }
  // this thread's rotary angle step (a constant table: read before the
  // dependency wait)
  __device__ __forceinline__ static uint64_t angle_step(const uint64_t* turn_fx, int ctid) {
    return turn_fx[ctid % R::HALF];
  }
  __device__ __forceinline__ void finish(long long pos, int n, uint64_t fx, float* q, int ctid) const {
    const int tb = ctid / R::HALF, i = ctid % R::HALF;
#pragma unroll
    for (int k = 0; k < R::K; ++k) {
      const int t = tb + k * R::RPP;
      if (t >= 16) continue;
      float a = 0.f, b = 0.f;
      if (t < n) {
        const float x1 = stored<bf16>(q1[k]), x2 = stored<bf16>(q2[k]);
        const float2 c = rope_cs(pos + t, fx);
        a = stored<bf16>(rot_lo(x1, x2, c));
        b = stored<bf16>(rot_hi(x1, x2, c));
      }
      q[t * QP + i] = a;
      q[t * QP + i + R::HALF] = b;
    }
  }
};

struct AkUnit {
  int sq, h, sp;
  long long k0, k1;  // keys [k0, k1) of the split that exist in this pass
  bool fresh;        // holds keys of the block (positions >= pos)
};

// Scores are kept in base 2: s2 = (q . k) / sqrt(Dh) * log2(e), so the
// softmax weights are exp2(s2 - max); partial maxima are stored back in
// natural units for the combine.
constexpr float AK_LOG2E = 1.4426950408889634f;
constexpr float AK_LN2 = 0.6931471805599453f;

template <typename Src, int DH, int MW, bool FUSED>
__global__ void __launch_bounds__(AkLayout<DH, MW>::THREADS, MW == 8 ? 1 : 2)
    attn_tma_kernel(Src src, int H, long long ctx_max, const uint64_t* __restrict__ turn_fx,
                    const float* __restrict__ qbuf,
                    const __grid_constant__ SeqRows sr, const __grid_constant__ SeqPtrs<bf16*> kcs,
                    const __grid_constant__ SeqPtrs<bf16*> vcs,
                    const __grid_constant__ SeqPtrs<const CUtensorMap*> kms,
                    const __grid_constant__ SeqPtrs<const CUtensorMap*> vms,
                    const __grid_constant__ SeqPtrs<evs_book*> books, int span, int nsplit_max,
                    const __grid_constant__ SeqPtrs<float*> part_os, const __grid_constant__ SeqPtrs<float*> part_mls,
                    const __grid_constant__ SeqPtrs<int*> arrivals, bf16* __restrict__ gout, int fold_cap) {
  using LY = AkLayout<DH, MW>;
  static_assert(FUSED == LY::MERGE_WARP, "the fused kernel runs with the merge warp");
  constexpr int NST = LY::NST;
  constexpr int QP = LY::QP;
  constexpr int MT = LY::MATH_THREADS;
  constexpr int KS = DH / 16;  // k-steps of Q K^T
  constexpr int NT = DH / 8;   // 8-dim output tiles
  extern __shared__ uint8_t ak_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(ak_raw) + 1023) & ~(uintptr_t)1023);
  float* q_s = reinterpret_cast<float*>(sm + LY::RING_B);                      // [16][QP]
  float* mw = reinterpret_cast<float*>(sm + LY::RING_B + LY::Q_B);             // [MW][16] max (base 2)
  float* lw = mw + MW * 16;                                                    // [MW][16] sum
  float* fw = lw + MW * 16;                                                    // [MW][16] merge weight
  float* ow = reinterpret_cast<float*>(sm + LY::RING_B + LY::Q_B + LY::ML_B);  // [MW][16][QP] O
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + LY::RING_B + LY::Q_B + LY::ML_B + LY::OW_B);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * NST + 1);
  int* fold_list = reinterpret_cast<int*>(sm + LY::FOLD_OFF);  // [fold_cap] (sequence << 16 | head)
  __shared__ long long s_pos[MAX_SEQ], s_tot[MAX_SEQ];
  __shared__ int s_act[MAX_SEQ], s_pref[MAX_SEQ + 1], s_nfold;
  const uint32_t ring = smem_u32(sm);
  const uint32_t bar0 = smem_u32(bars);
  auto full = [&](int s) { return bar0 + 8u * (uint32_t)s; };
  auto empty = [&](int s) { return bar0 + 8u * (uint32_t)(NST + s); };
  const uint32_t app = bar0 + 8u * (uint32_t)(2 * NST);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  pdl_trigger();
  if (tid == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), AK_GROUP_WARPS);  // the four warps of the group that took the stage
    }
    mbar_init(app, MT);
    *abort_flag = 0;
    s_nfold = 0;
    // committed lengths are fixed for the whole verify (commit runs after it)
    int acc = 0;
    for (int q = 0; q < sr.nseq; ++q) {
      const long long pos = books.p[q]->pos;
      const long long tot = min(pos + (long long)(sr.row0[q + 1] - sr.row0[q]), ctx_max);
      const int act = tot > 0 ? (int)min((tot + span - 1) / span, (long long)nsplit_max) : 0;
      s_pos[q] = pos;
      s_tot[q] = tot;
      s_act[q] = act;
      s_pref[q] = acc;
      acc += H * act;
    }
    s_pref[sr.nseq] = acc;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const int U = s_pref[sr.nseq];
  const int ub = (int)((long long)blockIdx.x * U / gridDim.x);
  const int ue = (int)((long long)(blockIdx.x + 1) * U / gridDim.x);
  auto decode = [&](int u) {
    int q = 0;
    while (u >= s_pref[q + 1]) ++q;
    const int r = u - s_pref[q], act = s_act[q];
    AkUnit x;
    x.sq = q;
    x.h = r / act;
    x.sp = r % act;
    x.k0 = (long long)x.sp * span;
    x.k1 = min(x.k0 + span, s_tot[q]);
    x.fresh = x.k1 > s_pos[q];
    return x;
  };
  auto nstages = [](const AkUnit& x) { return (int)((x.k1 - x.k0 + AK_STAGE - 1) / AK_STAGE); };
  // Processing order: the units of [ub, ue) without block keys, then those
  // with; (pass, u) = the current one, u == ue once past the end.
  auto advance = [&](int& pass, int& u) {
    for (;;) {
      if (++u >= ue) {
        if (pass == 1) {
          u = ue;
          return;
        }
        pass = 1;
        u = ub - 1;
        continue;
      }
      if ((int)decode(u).fresh == pass) return;
    }
  };
  constexpr int HT = MT + 32;  // math warps + merge warp
  if (LY::MERGE_WARP && warp == MW + 1) {
    // ---------------- merge warp: each unit's deposit -> the split's partial
    int pass = 0, u = ub - 1;
    advance(pass, u);
    if (u < ue) hand_arrive<2, HT>();  // the merge area starts free
    while (u < ue) {
      const AkUnit x = decode(u);
      const int n = sr.row0[x.sq + 1] - sr.row0[x.sq];
      int npass = pass, nu = u;
      advance(npass, nu);
      if (nu >= ue) break;  // the CTA's last unit: the math warps merge it themselves
      hand_wait<3, HT>();
      // per (row, warp): the warp's weight exp2(m_v - M), M the row's merged
      // max (0 for a warp that saw no key of the row)
      for (int q = lane; q < 16 * MW; q += 32) {
        const int t = q / MW, v = q % MW;
        float M = -INFINITY;
#pragma unroll
        for (int vv = 0; vv < MW; ++vv) M = fmaxf(M, mw[vv * 16 + t]);
        const float mv = mw[v * 16 + t];
        fw[v * 16 + t] = mv == -INFINITY ? 0.f : exp2f(mv - M);
      }
      __syncwarp();
      const bool good = !*abort_flag;
      float* part_o = part_os.p[x.sq];
      float* part_ml = part_mls.p[x.sq];
      if (good) {
        for (int e = lane; e < n * (DH / 4); e += 32) {
          const int t = e / (DH / 4), dd = 4 * (e % (DH / 4));
          const size_t base = ((size_t)x.h * nsplit_max + x.sp) * NTOK + t;
          merge_dims<MW, QP>(ow, fw, t, dd, part_o + base * DH + dd);
          if (dd == 0) {
            float M = -INFINITY, L = 0.f;
#pragma unroll
            for (int v = 0; v < MW; ++v) {
              M = fmaxf(M, mw[v * 16 + t]);
              L = fmaf(lw[v * 16 + t], fw[v * 16 + t], L);
            }
            part_ml[base * 2] = M * AK_LN2;
            part_ml[base * 2 + 1] = L;
          }
        }
      }
      __syncwarp();
      hand_arrive<2, HT>();  // the next unit may deposit
      if (FUSED && good) {
        // count the split; the last one of the head is folded after this
        // CTA's last unit
        __threadfence();
        __syncwarp();
        if (lane == 0) {
          int* cnt = arrivals.p[x.sq] + x.h;
          if (atomicAdd(cnt, 1) == s_act[x.sq] - 1) {
            __threadfence();  // the other splits' partials are read after this
            *cnt = 0;  // every split of the head has counted: ready for the next pass
            if (s_nfold < fold_cap) fold_list[s_nfold++] = (x.sq << 16) | x.h;
            else *abort_flag = 1;  // cannot happen with the host's capacity
          }
        }
      }
      pass = npass;
      u = nu;
    }
    hand_arrive<4, HT>();
    return;
  }

  if (warp == MW) {
    // ---------------- producer: one thread streams the CTA's stages
    if (lane != 0) return;
    const uint64_t pol = policy_evict_first();
    int gi = 0;
    bool ok = true, app_seen = false;
    int pass = 0, u = ub - 1;
    for (advance(pass, u); u < ue && ok; advance(pass, u)) {
      const AkUnit x = decode(u);
      if (x.fresh && !app_seen) {
        // the block's keys of this CTA's units are appended by now (by this
        // CTA, or by the rotary kernel before)
        if (FUSED) {
          if (!mbar_wait(app, 0, abort_flag)) {
            ok = false;
            break;
          }
        } else {
          pdl_wait();
        }
        app_seen = true;
      }
      const int y0 = (int)((long long)x.h * ctx_max + x.k0);
      const int nst = nstages(x);
      for (int st = 0; st < nst; ++st, ++gi) {
        const int s = gi % NST;
        if (gi >= NST && !mbar_wait(empty(s), (uint32_t)((gi / NST) - 1) & 1u, abort_flag)) {
          ok = false;
          break;
        }
        mbar_expect_tx(full(s), 2 * LY::TILE_B);
        const uint32_t kd = ring + (uint32_t)s * 2u * LY::TILE_B, vd = kd + LY::TILE_B;
#pragma unroll
        for (int hf = 0; hf < LY::HALVES; ++hf) {
          tma_load_2d(kd + hf * LY::BOX_B, kms.p[x.sq], full(s), hf * AK_BOX, y0 + st * AK_STAGE, pol);
          tma_load_2d(vd + hf * LY::BOX_B, vms.p[x.sq], full(s), hf * AK_BOX, y0 + st * AK_STAGE, pol);
        }
      }
    }
    // every issued copy lands before the CTA may exit (its shared memory is
    // their destination): wait for the last phase of each stage used
    volatile int no_abort = 0;
    for (int j = max(0, gi - NST); j < gi; ++j) mbar_wait_slow(full(j % NST), (uint32_t)(j / NST) & 1u, &no_abort);
    return;
  }

  // ---------------- math warps
  const int ctid = tid;  // 0 .. MT - 1
  const int gp = warp / AK_GROUP_WARPS, wg = warp % AK_GROUP_WARPS;
  const int g = lane >> 2, t4 = lane & 3;
  const int d = H * DH;
  int pass = 0, u = ub - 1;
  advance(pass, u);  // the first unit in processing order
  const uint64_t fx = FUSED ? QueryRows<Src, DH, QP, MT>::angle_step(turn_fx, ctid) : 0;
  pdl_wait();
  QueryRows<Src, DH, QP, MT> qr;
  int cur_h = -1, cur_sq = -1;
  // the rotated queries of head h: rotated here (FUSED) or by the rotary
  // kernel before (rows in qbuf [rows][H][DH], already rounded to bf16)
  auto queries = [&](const AkUnit& x) {
    const int n = sr.row0[x.sq + 1] - sr.row0[x.sq], r0 = sr.row0[x.sq];
    if (FUSED) {
      qr.load(src, x.h, r0, n, ctid);
      qr.finish(s_pos[x.sq], n, QueryRows<Src, DH, QP, MT>::angle_step(turn_fx, ctid), q_s, ctid);
    } else {
      for (int e = ctid; e < 16 * DH; e += MT) {
        const int t = e / DH, dd = e % DH;
        q_s[t * QP + dd] = t < n ? qbuf[((size_t)(r0 + t) * H + x.h) * DH + dd] : 0.f;
      }
    }
  };
  if (!FUSED) {
    if (u < ue) {
      const AkUnit x = decode(u);
      queries(x);
      cur_h = x.h;
      cur_sq = x.sq;
    }
  } else {
  // the first unit's queries load while the block's keys are appended
  if (u < ue) {
    const AkUnit x = decode(u);
    qr.load(src, x.h, sr.row0[x.sq], sr.row0[x.sq + 1] - sr.row0[x.sq], ctid);
  }
  if (blockIdx.x == 0 && ctid < sr.nseq) {
    const int q = ctid;
    if (s_pos[q] + (sr.row0[q + 1] - sr.row0[q]) > ctx_max) set_status(books.p[q], EVS_DEV_KV_OVERFLOW);
  }
  // rotate and append the block's keys / values of this CTA's fresh units
  for (int v = ub; v < ue; ++v) {
    const AkUnit x = decode(v);
    if (!x.fresh) continue;
    const long long pos = s_pos[x.sq];
    const int t0 = (int)(max(x.k0, pos) - pos), t1 = (int)(x.k1 - pos);
    append_rows<Src, DH, MT>(src, d, x.h, sr.row0[x.sq], pos, t0, t1, ctx_max, fx, kcs.p[x.sq], vcs.p[x.sq], ctid);
  }
  // the producer's tensor-map loads (async proxy) read these rows next
  asm volatile("fence.proxy.async.global;" ::: "memory");
  mbar_arrive(app);
  if (u < ue) {
    const AkUnit x = decode(u);
    qr.finish(s_pos[x.sq], sr.row0[x.sq + 1] - sr.row0[x.sq], fx, q_s, ctid);
    cur_h = x.h;
    cur_sq = x.sq;
  }
  }
  math_sync<MT>();

  int gi = 0;  // ring stages so far
  bool ok = true;
  const float c2 = rsqrtf((float)DH) * AK_LOG2E;
  int last_sq = -1, last_h = 0;  // the last unit, when the math warps merged it
  for (; u < ue; advance(pass, u)) {
    const AkUnit x = decode(u);
    const int n = sr.row0[x.sq + 1] - sr.row0[x.sq], r0 = sr.row0[x.sq];
    int lpass = pass, lu = u;
    advance(lpass, lu);
    const bool last = lu >= ue;
    const long long pos = s_pos[x.sq];
    if (x.h != cur_h || x.sq != cur_sq) {
      queries(x);
      math_sync<MT>();
      cur_h = x.h;
      cur_sq = x.sq;
    }
    // Q as the A operand: rows g and g + 8 (queries past n are zero)
    uint32_t qa[KS][4];
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
      const int c0 = kk * 16 + 2 * t4;
      const float2 a0 = *reinterpret_cast<const float2*>(q_s + g * QP + c0);
      const float2 a1 = *reinterpret_cast<const float2*>(q_s + (g + 8) * QP + c0);
      const float2 a2 = *reinterpret_cast<const float2*>(q_s + g * QP + c0 + 8);
      const float2 a3 = *reinterpret_cast<const float2*>(q_s + (g + 8) * QP + c0 + 8);
      qa[kk][0] = pack_bf16x2(a0.x, a0.y);
      qa[kk][1] = pack_bf16x2(a1.x, a1.y);
      qa[kk][2] = pack_bf16x2(a2.x, a2.y);
      qa[kk][3] = pack_bf16x2(a3.x, a3.y);
    }
    float o[NT][4];
#pragma unroll
    for (int jj = 0; jj < NT; ++jj) o[jj][0] = o[jj][1] = o[jj][2] = o[jj][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // rows g, g + 8 (base-2 max)
    // keys relative to pos: row r sees keys with rel <= r; the split ends at rel kend
    const int kend = (int)(x.k1 - pos);
    const int nst = (int)((x.k1 - x.k0 + AK_STAGE - 1) / AK_STAGE);
    for (int st = gp; st < nst; st += LY::GROUPS) {
      const int gs = gi + st, s = gs % NST;
      if (ok) ok = __all_sync(0xffffffffu, wait_inl(full(s), (uint32_t)(gs / NST) & 1u, abort_flag));
      const int kw = (int)(x.k0 + (long long)st * AK_STAGE - pos) + 16 * wg;  // this warp's first key, relative
      const uint32_t kb = ring + (uint32_t)s * 2u * LY::TILE_B, vb = kb + LY::TILE_B;
      if (ok && kw < kend) {
        if (kw + 16 > kend) {
          // rows of this warp past the split's end: V zeroed (K is masked)
          const int z0 = kend - kw, zr = 16 - z0;
          for (int e = lane; e < zr * 8 * LY::HALVES; e += 32) {
            const int hf = e / (zr * 8), rem = e % (zr * 8);
            const int r = 16 * wg + z0 + rem / 8;
            *reinterpret_cast<uint4*>(sm + (size_t)s * 2 * LY::TILE_B + LY::TILE_B + hf * LY::BOX_B + r * 128 +
                                      (rem % 8) * 16) = make_uint4(0u, 0u, 0u, 0u);
          }
          // ordered before the next tensor-map load into this stage
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
        }
        // S = Q K^T for 16 keys: two 8-key tiles
        float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
          const int mi = lane >> 3;
          const int r = 16 * wg + ((mi >> 1) << 3) + (lane & 7);
          const int c = 2 * kk + (mi & 1);
          uint32_t b[4];
          ldsm4(kb + tile_off(r, c, LY::BOX_B), b);
          mma16816(sc[0], qa[kk], b[0], b[1]);
          mma16816(sc[1], qa[kk], b[2], b[3]);
        }
        float mx0, mx1;
        if (kw + 15 < 0 && kw + 16 <= kend) {
          // committed keys, all inside the split: every row sees all 16
#pragma unroll
          for (int jj = 0; jj < 2; ++jj)
#pragma unroll
            for (int e = 0; e < 4; ++e) sc[jj][e] *= c2;
          mx0 = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
          mx1 = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));
        } else {
          mx0 = mx1 = -INFINITY;
#pragma unroll
          for (int jj = 0; jj < 2; ++jj)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int key = kw + 8 * jj + 2 * t4 + (e & 1);
              const bool in = key < kend && key <= ((e >> 1) ? g + 8 : g);
              sc[jj][e] = in ? sc[jj][e] * c2 : -INFINITY;
              if (e >> 1)
                mx1 = fmaxf(mx1, sc[jj][e]);
              else
                mx0 = fmaxf(mx0, sc[jj][e]);
            }
        }
#pragma unroll
        for (int xo = 1; xo < 4; xo <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, xo));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, xo));
        }
        // The running max moves only when a score exceeds it by more than
        // 2^8 (weights stay <= 256); the final normalisation divides the
        // common factor out.  A row with no visible key yet keeps
        // (max, sum, output) = (-inf, 0, 0).
        const float n0r = mx0 > m0 + 8.f ? mx0 : m0, n1r = mx1 > m1 + 8.f ? mx1 : m1;
        const float b0 = n0r == -INFINITY ? 0.f : n0r, b1 = n1r == -INFINITY ? 0.f : n1r;
        const float a0 = n0r == m0 ? 1.f : exp2f(m0 - b0), a1 = n1r == m1 ? 1.f : exp2f(m1 - b1);
        m0 = n0r;
        m1 = n1r;
        float p[2][4];
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
          p[jj][0] = exp2f(sc[jj][0] - b0);
          p[jj][1] = exp2f(sc[jj][1] - b0);
          p[jj][2] = exp2f(sc[jj][2] - b1);
          p[jj][3] = exp2f(sc[jj][3] - b1);
        }
        l0 = fmaf(l0, a0, (p[0][0] + p[0][1]) + (p[1][0] + p[1][1]));
        l1 = fmaf(l1, a1, (p[0][2] + p[0][3]) + (p[1][2] + p[1][3]));
        if (__any_sync(0xffffffffu, a0 != 1.f || a1 != 1.f)) {
#pragma unroll
          for (int jj = 0; jj < NT; ++jj) {
            o[jj][0] *= a0;
            o[jj][1] *= a0;
            o[jj][2] *= a1;
            o[jj][3] *= a1;
          }
        }
        // O += P V: P (16 queries x 16 keys) as the A operand
        const uint32_t pa[4] = {pack_bf16x2(p[0][0], p[0][1]), pack_bf16x2(p[0][2], p[0][3]),
                                pack_bf16x2(p[1][0], p[1][1]), pack_bf16x2(p[1][2], p[1][3])};
#pragma unroll
        for (int jd = 0; jd < NT; jd += 2) {
          const int mi = lane >> 3;
          const int r = 16 * wg + ((mi & 1) << 3) + (lane & 7);
          const int c = jd + (mi >> 1);
          uint32_t b[4];
          ldsm4_t(vb + tile_off(r, c, LY::BOX_B), b);
          mma16816(o[jd], pa, b[0], b[1]);
          mma16816(o[jd + 1], pa, b[2], b[3]);
        }
      }
      __syncwarp();
      if (ok && lane == 0) mbar_arrive(empty(s));
    }
    gi += nst;
    // row sums over the quad, then (max, sum, O) into the merge area for the
    // merge warp
#pragma unroll
    for (int xo = 1; xo < 4; xo <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, xo);
      l1 += __shfl_xor_sync(0xffffffffu, l1, xo);
    }
    if (LY::MERGE_WARP) hand_wait<2, HT>();
    if (t4 == 0) {
      mw[warp * 16 + g] = m0;
      mw[warp * 16 + g + 8] = m1;
      lw[warp * 16 + g] = l0;
      lw[warp * 16 + g + 8] = l1;
    }
#pragma unroll
    for (int jj = 0; jj < NT; ++jj) {
      float* q0 = ow + ((size_t)warp * 16 + g) * QP + 8 * jj + 2 * t4;
      *reinterpret_cast<float2*>(q0) = make_float2(o[jj][0], o[jj][1]);
      *reinterpret_cast<float2*>(q0 + 8 * QP) = make_float2(o[jj][2], o[jj][3]);
    }
    if (LY::MERGE_WARP && !last) {
      hand_arrive<3, HT>();
      continue;
    }
    // without a merge warp, and for the CTA's last unit (the merge warp
    // would be the tail): the math warps merge the unit in warp order
    math_sync<MT>();
    if (ctid < 16 * MW) {
      const int t = ctid / MW, v = ctid % MW;
      float M = -INFINITY;
#pragma unroll
      for (int vv = 0; vv < MW; ++vv) M = fmaxf(M, mw[vv * 16 + t]);
      const float mv = mw[v * 16 + t];
      fw[v * 16 + t] = mv == -INFINITY ? 0.f : exp2f(mv - M);
    }
    math_sync<MT>();
    if (ok) {
      float* part_o = part_os.p[x.sq];
      float* part_ml = part_mls.p[x.sq];
      for (int e = ctid; e < n * (DH / 4); e += MT) {
        const int t = e / (DH / 4), dd = 4 * (e % (DH / 4));
        const size_t base = ((size_t)x.h * nsplit_max + x.sp) * NTOK + t;
        merge_dims<MW, QP>(ow, fw, t, dd, part_o + base * DH + dd);
        if (dd == 0) {
          float M = -INFINITY, L = 0.f;
#pragma unroll
          for (int v = 0; v < MW; ++v) {
            M = fmaxf(M, mw[v * 16 + t]);
            L = fmaf(lw[v * 16 + t], fw[v * 16 + t], L);
          }
          part_ml[base * 2] = M * AK_LN2;
          part_ml[base * 2 + 1] = L;
        }
      }
    }
    if (LY::MERGE_WARP) {
      __threadfence();  // the partial is visible before the split is counted
      last_sq = x.sq;
      last_h = x.h;
    }
    math_sync<MT>();  // the merge area is rewritten by the next unit
  }
  if (!LY::MERGE_WARP) {
    if (!ok && ctid == 0)
      for (int q = 0; q < sr.nseq; ++q) set_status(books.p[q], EVS_DEV_TIMEOUT);
    return;
  }
  // every unit merged and counted; the heads whose last split finished here
  // are folded: per query row t the splits holding keys <= its position,
  // their weights exp(m_c - M) and l_c (the merge area is free: [16][64]
  // each, then the row sums [16]), all loads of a phase in flight
  hand_wait<4, HT>();
  if (last_sq >= 0 && ctid == 0 && !*abort_flag) {
    // count the last split (after the merge warp's counts: one writer of the
    // fold list at a time)
    int* cnt = arrivals.p[last_sq] + last_h;
    if (atomicAdd(cnt, 1) == s_act[last_sq] - 1) {
      __threadfence();
      *cnt = 0;
      if (s_nfold < fold_cap) fold_list[s_nfold++] = (last_sq << 16) | last_h;
      else *abort_flag = 1;
    }
  }
  math_sync<MT>();
  for (int f = 0; f < s_nfold; ++f) {
    const int sq = fold_list[f] >> 16, h = fold_list[f] & 0xffff;
    const int n = sr.row0[sq + 1] - sr.row0[sq], r0 = sr.row0[sq];
    const long long pos = s_pos[sq];
    __threadfence();
    float* wt = ow;
    float* lc = ow + 16 * ATTN_SPLITS_MAX;
    float* lt = lc + 16 * ATTN_SPLITS_MAX;
    const float* pml = part_mls.p[sq] + ((size_t)h * nsplit_max) * NTOK * 2;
    const float* po = part_os.p[sq] + ((size_t)h * nsplit_max) * NTOK * DH;
    for (int tb = 0; tb < 16; tb += MT / 16) {
      const int t = tb + (ctid >> 4), l16 = ctid & 15;  // 16 threads per row, every lane shuffles
      const int nc = t < n ? (int)(min(pos + t, ctx_max - 1) / span) + 1 : 0;
      float2 ml[ATTN_SPLITS_MAX / 16];
      float M = -INFINITY;
#pragma unroll
      for (int k = 0; k < ATTN_SPLITS_MAX / 16; ++k) {
        const int c = l16 + 16 * k;
        ml[k] = c < nc ? __ldcg(reinterpret_cast<const float2*>(pml + ((size_t)c * NTOK + t) * 2))
                       : make_float2(-INFINITY, 0.f);
        M = fmaxf(M, ml[k].x);
      }
#pragma unroll
      for (int xo = 8; xo > 0; xo >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, xo));
#pragma unroll
      for (int k = 0; k < ATTN_SPLITS_MAX / 16; ++k) {
        const int c = l16 + 16 * k;
        if (c < nc) {
          wt[t * ATTN_SPLITS_MAX + c] = ml[k].x == -INFINITY ? 0.f : expf(ml[k].x - M);
          lc[t * ATTN_SPLITS_MAX + c] = ml[k].y;
        }
      }
    }
    math_sync<MT>();
    // outputs four dims per item (a thread holds at most two), each summed
    // over the splits in order; the last 16 threads, which hold one item
    // when there are fewer than 2 MT, then take the rows' l = sum_c w_c l_c
    // in split order, and the quotients wait for those
    static_assert(!FUSED || 16 * (DH / 4) <= 2 * MT, "at most two output items per thread");
    const int items = n * (DH / 4);
    float4 o[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      o[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      const int e = ctid + k * MT;
      if (e >= items) continue;
      const int t = e / (DH / 4), d4 = 4 * (e % (DH / 4));
      const int nc = (int)(min(pos + t, ctx_max - 1) / span) + 1;
#pragma unroll 16
      for (int c = 0; c < nc; ++c) {
        const float w = wt[t * ATTN_SPLITS_MAX + c];
        const float4 oc = __ldcg(reinterpret_cast<const float4*>(po + ((size_t)c * NTOK + t) * DH + d4));
        if (w != 0.f) {
          o[k].x = fmaf(oc.x, w, o[k].x);
          o[k].y = fmaf(oc.y, w, o[k].y);
          o[k].z = fmaf(oc.z, w, o[k].z);
          o[k].w = fmaf(oc.w, w, o[k].w);
        }
      }
    }
    if (ctid >= MT - 16 && ctid - (MT - 16) < n) {
      const int t = ctid - (MT - 16);
      const int nc = (int)(min(pos + t, ctx_max - 1) / span) + 1;
      float l = 0.f;
      for (int c = 0; c < nc; ++c) {
        const float w = wt[t * ATTN_SPLITS_MAX + c];
        if (w != 0.f) l = fmaf(lc[t * ATTN_SPLITS_MAX + c], w, l);
      }
      lt[t] = l;
    }
    math_sync<MT>();
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int e = ctid + k * MT;
      if (e >= items) continue;
      const int t = e / (DH / 4), d4 = 4 * (e % (DH / 4));
      store_out4(gout + (size_t)(r0 + t) * H * DH + h * DH + d4, o[k], lt[t]);
    }
    math_sync<MT>();  // the area is rewritten by the next fold
  }
  if (!ok && ctid == 0)
    for (int q = 0; q < sr.nseq; ++q) set_status(books.p[q], EVS_DEV_TIMEOUT);
}

template <typename Src, int DH, int MW, bool FUSED>
cudaError_t attn_tma_launch_t(const LaunchCtx& L, Src s, int H, const SeqRows& sr, long long ctx_max,
                              const AttnSeq& as, const AttnBufs& B, void* g) {
  using LY = AkLayout<DH, MW>;
  auto k = attn_tma_kernel<Src, DH, MW, FUSED>;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const long long units = (long long)sr.nseq * H * B.nsplit_max;
  const int grid = (int)std::max(1LL, std::min<long long>(units, (long long)sms * (MW == 8 ? 1 : 2)));
  // a CTA folds at most the heads of its own units
  const int fold_cap = (int)((units + grid - 1) / grid) + 1;
  const size_t smem = LY::SMEM + sizeof(int) * fold_cap;
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  SeqPtrs<bf16*> kc{}, vc{};
  SeqPtrs<const CUtensorMap*> km{}, vm{};
  for (int b = 0; b < sr.nseq; ++b) {
    kc.p[b] = (bf16*)as.kc.p[b];
    vc.p[b] = (bf16*)as.vc.p[b];
    km.p[b] = as.kmap.p[b];
    vm.p[b] = as.vmap.p[b];
  }
  return launch(L, k, dim3(grid), dim3(LY::THREADS), smem, s, H, ctx_max, (const uint64_t*)B.turn_fx,
                (const float*)B.qbuf, sr, kc, vc, km,
                vm, as.book, B.span, B.nsplit_max, as.part_o, as.part_ml, as.arrivals, (bf16*)g, fold_cap);
}

template <typename Src>
cudaError_t attn_tma_dh(const LaunchCtx& L, Src s, int H, int Dh, const SeqRows& sr, long long ctx_max,
                        const AttnSeq& as, const AttnBufs& B, void* g, bool fused) {
  // the configuration is a function of the cache size alone (the caller's
  // choice of fused), so every pass over a cache rounds alike
  switch (Dh) {
    case 64:
      return fused ? attn_tma_launch_t<Src, 64, 8, true>(L, s, H, sr, ctx_max, as, B, g)
                   : attn_tma_launch_t<Src, 64, 4, false>(L, s, H, sr, ctx_max, as, B, g);
    case 128:
      return fused ? attn_tma_launch_t<Src, 128, 8, true>(L, s, H, sr, ctx_max, as, B, g)
                   : attn_tma_launch_t<Src, 128, 4, false>(L, s, H, sr, ctx_max, as, B, g);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

bool attn_tma_eligible(int dtype, int H, int Dh, long long ctx_max) {
  return dtype == EVS_BF16 && (Dh == 64 || Dh == 128) && (long long)H * ctx_max + AK_STAGE < (1LL << 31);
}

cudaError_t launch_attn_tma(const LaunchCtx& L, MixSrc src, int H, int Dh, const SeqRows& sr, long long ctx_max,
                            const AttnSeq& as, const AttnBufs& B, void* g, bool fused) {
  for (int b = 0; b < sr.nseq; ++b)
    if (!as.kmap.p[b] || !as.vmap.p[b] || (fused && !as.arrivals.p[b])) return cudaErrorInvalidValue;
  if (B.span % AK_STAGE || B.nsplit_max > ATTN_SPLITS_MAX) return cudaErrorInvalidValue;
  if (src.ws) return attn_tma_dh(L, SrcSlots{src.ws, src.tab, src.slot_rows}, H, Dh, sr, ctx_max, as, B, g, fused);
  if (src.f32)
    return attn_tma_dh(L, SrcPlain<float>{(const float*)src.p, src.ld}, H, Dh, sr, ctx_max, as, B, g, fused);
  return attn_tma_dh(L, SrcPlain<bf16>{(const bf16*)src.p, src.ld}, H, Dh, sr, ctx_max, as, B, g, fused);
}

bool encode_kv_maps(CUtensorMap* kmap, CUtensorMap* vmap, const void* kc, const void* vc, int H, int Dh,
                    long long ctx_max, char* err, size_t errlen) {
  const uint64_t rows = (uint64_t)H * (uint64_t)ctx_max;
  return encode_tmap_2d(kmap, kc, (uint64_t)Dh, rows, AK_BOX, AK_STAGE, err, errlen) &&
         encode_tmap_2d(vmap, vc, (uint64_t)Dh, rows, AK_BOX, AK_STAGE, err, errlen);
}

}  // namespace evs
