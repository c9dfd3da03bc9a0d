// C ABI of libevs: model / state ownership, the verify sequence, CUDA-graph
// capture, accept / commit entry points and the single-operator entry points.
//
// The verify sequence is the EvSpark block-verification forward pass
// (preprint abstract, contribution (i); discussion post, "What we
// implemented"): one pass over n = gamma'+1 tokens through every layer, each
// mixer writing the state after every block position to its spare bank.
// Commit (same passages: "sliced directly to the accepted boundary") flips
// banks on the device; nothing is recomputed or copied.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "evs_internal.cuh"

using namespace evs;

namespace {

thread_local std::string g_err;
std::atomic<long long> g_launches{0};
std::atomic<unsigned long long> g_state_uid{0};

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return code;
}

#define CUDA_TRY(x)                                                                                 \
  do {                                                                                              \
    cudaError_t e_ = (x);                                                                           \
    if (e_ != cudaSuccess)                                                                          \
      return fail(EVS_ERR_CUDA, "%s failed: %s (%s:%d)", #x, cudaGetErrorString(e_), __FILE__, __LINE__); \
  } while (0)

#define EVS_TRY(x)          \
  do {                      \
    int r_ = (x);           \
    if (r_ != EVS_OK) return r_; \
  } while (0)

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

int num_sms_current(int* out) {
  int dev = 0;
  CUDA_TRY(cudaGetDevice(&dev));
  CUDA_TRY(cudaDeviceGetAttribute(out, cudaDevAttrMultiProcessorCount, dev));
  return EVS_OK;
}

struct LayerW {
  int kind, param;
  const void *w_in, *w_out, *w_gu, *w_down;
  const float *taps, *lam, *res;
  CUtensorMap m_in, m_out, m_gu, m_down;
  const uint8_t *pk_in, *pk_out, *pk_gu, *pk_down;  // packed copies (bf16), in wpack
};

struct LayerS {
  float* ring;   // FIR inputs [L-1+n_max][d], position p at row p mod (L-1+n_max)
  float* st[2];
  void* kc;
  void* vc;
  const CUtensorMap* kmap;  // device tensor maps of kc / vc (bf16 caches), else null
  const CUtensorMap* vmap;
};

struct GraphEntry {
  // key
  int n, mode, top_k;
  float T;
  const void *tok, *logits, *p, *q, *u, *acc, *otok;
  bool round;
  bool host_io;  // evs_round_host: the copies to and from the staging are in the graph
  // batched rounds: the sequences' states (by creation id, never reused)
  // and block lengths
  int nseq;
  unsigned long long uid[MAX_SEQ];
  int ns[MAX_SEQ];
  // value
  cudaGraphExec_t exec;
  int kernels;
  unsigned long long last_use;
};

}  // namespace

void evs::count_launch(int k) { g_launches += k; }

struct evs_model {
  evs_config cfg;
  std::vector<int> kind, param;
  int num_sms;
  bool tc;  // bf16 storage: tensor-core GEMMs
  const void* embed;
  const void* head;
  CUtensorMap m_head;
  const uint8_t* pk_head;
  uint8_t* wpack;  // library-owned packed projection weights (bf16), or null
  std::vector<LayerW> L;
  Partials p_in, p_out, p_gu, p_down, p_head;  // with device slot tables
  // the same five as stream-K plans over the same unit ranges (a cluster
  // plan of cl ranks per tile becomes cl stream-K contributors per tile, so
  // the packed weight order is unchanged): passes of more than 16 rows
  Partials q_in, q_out, q_gu, q_down, q_head;
  int4* tab_dev;                               // the ten slot tables
  size_t ws_bytes;                             // largest partial workspace
  bool has_attn;
  // bf16: projection weights repacked (library copy in wpack) with the
  // gate/up rows interleaved for the SwiGLU column order
  bool packed;
  // Opt-in fusions of the small elementwise kernels into the GEMMs (packed
  // weights only), bit-identical to the separate kernels:
  //  swiglu (EVS_OPT_SWIGLU_EPILOGUE): the gate/up GEMM applies SiLU-and-multiply in
  //    its epilogue (no activation kernel);
  //  fuse (EVS_OPT_NORM_IN_GEMM): the GEMMs that read RMSNorm output build their B
  //    tiles from the fp32 residual rows (no normalisation kernels).
  // Both measured slower on the 7B-shaped stack: with a small kernel in
  // between, the next GEMM's CTAs are resident and loading weights before
  // their inputs are ready, which hides more than the kernel costs; the
  // converter also adds start-up latency and its larger blocks keep the next
  // mixer from starting early.
  bool swiglu;
  bool fuse;
  // stream-K in-projection and gate/up GEMMs leave their partial slots to
  // the consuming mixer / activation kernel (GEMM_SLOTS): no fixup tail
  // (bf16; EVS_OPT_GEMM_SUMS_SLOTS keeps the GEMM-side fixup)
  bool slots;
  // out / down GEMMs too (stream-K on every SM instead of cluster split-K),
  // the residual add and its sums of squares done by resid_norm (fused
  // converters: the GEMM's own residual epilogue, on the same split)
  bool slots_resid;
  int n_max;
};

struct evs_state {
  evs_model* m;
  unsigned long long uid;  // creation id (graph keys of batched rounds)
  long long ctx_max;
  evs_book* book;
  int host_pos;
  bool host_pos_known;
  int host_pending;
  float* X;
  void *xn, *g, *h;
  // work buffers hold ROWS_MAX token rows (a batched pass over several
  // sequences' blocks uses the first state's)
  float* fin;   // [ROWS_MAX][max(3d, 2F, V)] final GEMM sums (mixer / MLP inputs)
  float* pout;  // [NTOK][max(3d, 2F, V)]: GEMM outputs of evs_profile_gemms
  float* ss;    // [tiles of d][ROWS_MAX] per-tile sums of squares
  int* cnt;     // [max tiles] GEMM arrival counters
  int cnt_len;
  // evs_round_host: the block's tokens [NTOK] and the result (accepted,
  // token) on the device, and their pinned host staging [NTOK + 2]
  int32_t* io_dev = nullptr;
  int32_t* io_pinned = nullptr;
  float* ws[2];
  void* attn_scratch;
  AttnBufs ab;
  std::vector<LayerS> S;
  CUtensorMap m_xn, m_g, m_h;
  CUtensorMap m_xf;  // fp32 X [ROWS_MAX][d] (RMSNorm converter source, 16-row boxes)
  bool use_graphs, pdl;
  int pf_units;  // next-weight L2 prefetch per CTA (units of 128x64)
  cudaStream_t cap;
  // Persistent engine (single-sequence bf16 verifies): the phase program,
  // its counters and the spans it is cut into by the attention mixers
  struct EngSeg {
    int ph0, ph1;
    int attn_layer;   // the attention layer whose mixer follows the span, or -1
    float* attn_ws;   // that layer's in-projection slots
  };
  bool engine_ok = false;
  bool use_engine = false;
  EngPhase* eng_prog = nullptr;
  std::vector<EngSeg> eng_segs;
  int* eng_cnt = nullptr;
  size_t eng_cnt_bytes = 0;
  int eng_row_floats = 0;
  std::vector<GraphEntry> graphs;
  unsigned long long tick;
  std::vector<void*> allocs;
  size_t alloc_bytes = 0;
};

namespace {

size_t esize(int dtype) { return dtype == EVS_BF16 ? 2 : 4; }

// Fault injection for tests: EVS_ALLOC_LIMIT=<bytes> caps one state's
// device allocations; beyond it dmalloc reports EVS_ERR_OOM without
// allocating (the same path a real cudaMalloc failure takes).
size_t alloc_limit() {
  const char* v = getenv("EVS_ALLOC_LIMIT");
  return v ? (size_t)strtoull(v, nullptr, 10) : 0;
}

int dmalloc(evs_state* s, void** p, size_t bytes) {
  if (bytes == 0) bytes = 16;
  const size_t lim = alloc_limit();
  if (lim && s->alloc_bytes + bytes > lim)
    return fail(EVS_ERR_OOM, "allocation of %zu bytes exceeds EVS_ALLOC_LIMIT (%zu in use)", bytes, s->alloc_bytes);
  cudaError_t e = cudaMalloc(p, bytes);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(EVS_ERR_OOM, "cudaMalloc(%zu) failed: %s", bytes, cudaGetErrorString(e));
  }
  s->allocs.push_back(*p);
  s->alloc_bytes += bytes;
  return EVS_OK;
}

// ------------------------------------------------------------------ engine
// Whether the persistent engine can run this model: the bf16 packed path with
// every stream-K GEMM leaving slots to its consumers, FIR filters of at most
// 128 taps, and the head's stream-K view over its cluster plan.
// The stream-K plan the engine runs a weight matrix with: the plan itself,
// or for a cluster plan its stream-K twin, which gives every CTA the same
// units (so the packed order is the same) and sums the same partials in the
// same order (cluster ranks = slots).
static const Partials& eng_plan(const Partials& p, const Partials& q) { return p.cl == 0 ? p : q; }

static bool engine_eligible(const evs_model* m) {
  const evs_config& c = m->cfg;
  if (!(m->tc && m->packed && m->slots && m->slots_resid) || m->fuse || m->swiglu) return false;
  const Partials& pin = eng_plan(m->p_in, m->q_in);
  const Partials& pout = eng_plan(m->p_out, m->q_out);
  const Partials& pgu = eng_plan(m->p_gu, m->q_gu);
  const Partials& pdn = eng_plan(m->p_down, m->q_down);
  const Partials& phd = eng_plan(m->p_head, m->q_head);
  if (pin.max_cnt > SLOTS_MIX_MAX || pgu.max_cnt > SLOTS_MIX_MAX || pout.max_cnt > SLOTS_RESID_MAX ||
      pdn.max_cnt > SLOTS_RESID_MAX || phd.max_cnt > 8)
    return false;
  const Partials* all[5] = {&pin, &pout, &pgu, &pdn, &phd};
  const Partials* own[5] = {&m->p_in, &m->p_out, &m->p_gu, &m->p_down, &m->p_head};
  for (int k = 0; k < 5; ++k)
    if (all[k]->G > m->num_sms || all[k]->G != own[k]->G || all[k]->U != own[k]->U) return false;
  if (c.d_model % TILE_M || c.d_model / TILE_M > RESID_TILES_ROW || c.d_ffn % TILE_K || c.vocab % TILE_M) return false;
  for (const LayerW& L : m->L)
    if (L.kind == EVS_LAYER_FIR && L.param > 128) return false;
  return true;
}

// The phase program of a state: every GEMM and row phase of a verify in
// order, cut into spans at the attention mixers.  cnt == nullptr counts the
// counters the program needs (*ncnt) without building it.
static void engine_program(evs_state* s, int* cnt, std::vector<EngPhase>* out, std::vector<evs_state::EngSeg>* segs,
                           size_t* ncnt, int* row_floats) {
  const evs_model* m = s->m;
  const evs_config& c = m->cfg;
  const int d = c.d_model, F = c.d_ffn, V = c.vocab;
  size_t k = 0;
  auto take = [&](int n) -> int* {
    int* p = cnt ? cnt + k : nullptr;
    k += n;
    return p;
  };
  int wsi = 0;
  std::vector<EngPhase>& ph = *out;
  ph.clear();
  segs->clear();
  *row_floats = 0;
  auto gemm = [&](const Partials& P, const uint8_t* wpk, int bmap, int* ready, int target) -> EngPhase& {
    EngPhase e{};
    e.kind = ENG_GEMM;
    e.G = P.G;
    e.KB = P.KB;
    e.T = (P.N + TILE_M - 1) / TILE_M;
    e.U = P.U;
    e.bmap = bmap;
    e.target = ready ? target : 0;
    e.wpk = wpk;
    e.tab = P.tab;
    e.ws = s->ws[(wsi++) & 1];
    e.cnt = take(e.T);
    e.ready = ready;
    ph.push_back(e);
    return ph.back();
  };
  auto row = [&](int kind, int items, const EngPhase& src) -> EngPhase& {
    EngPhase e{};
    e.kind = kind;
    e.G = items;
    e.tab = src.tab;
    e.ws = src.ws;
    e.cnt = src.cnt;
    e.ready = take(1);
    ph.push_back(e);
    return ph.back();
  };
  // residual add + RMSNorm after an out / down GEMM (one item per 128-column
  // tile); returns the counter the normalised tiles raise
  auto resid_norm = [&](const EngPhase& g) -> int* {
    EngPhase& r = row(ENG_RESID, d / TILE_M, g);
    r.done = take(1);
    r.X = s->X;
    r.ss = s->ss;
    r.out = s->xn;
    r.out_ld = d;
    return r.ready;
  };
  int* xn_ready = nullptr;  // the first in-projection reads the embedding kernel's rows
  int seg0 = 0;
  int* g_ready = nullptr;
  int g_target = 0;
  for (size_t i = 0; i < m->L.size(); ++i) {
    const LayerW& w = m->L[i];
    const LayerS& st = s->S[i];
    EngPhase in = gemm(eng_plan(m->p_in, m->q_in), w.pk_in, ENG_B_XN, xn_ready, d / TILE_M);
    if (w.kind == EVS_LAYER_ATTN) {
      segs->push_back({seg0, (int)ph.size(), (int)i, in.ws});
      seg0 = (int)ph.size();
      g_ready = nullptr;  // the attention kernels finish before the next span starts
      g_target = 0;
    } else {
      const bool fir = w.kind == EVS_LAYER_FIR;
      // IIR items take two blocks of 256 / M channels when one block each
      // would leave CTAs with two items
      const int cpb = fir ? 32 : 256 / w.param;
      const int sub = !fir && d / cpb > m->num_sms && d % (2 * cpb) == 0 && 2 * cpb <= TILE_M ? 2 : 1;
      const int items = d / (cpb * sub);
      EngPhase& mx = row(fir ? ENG_FIR : ENG_IIR, items, in);
      mx.L = w.param;
      mx.sub = sub;
      mx.p0 = fir ? w.taps : w.lam;
      mx.p1 = fir ? nullptr : w.res;
      mx.bank0 = fir ? st.ring : st.st[0];
      mx.bank1 = fir ? nullptr : st.st[1];
      mx.ring = fir ? w.param - 1 + m->n_max : 0;
      mx.out = s->g;
      mx.out_ld = d;
      g_ready = mx.ready;
      g_target = items;
      *row_floats = std::max(*row_floats, engine_row_floats(mx.kind, w.param, sub));
    }
    EngPhase out_g = gemm(eng_plan(m->p_out, m->q_out), w.pk_out, ENG_B_G, g_ready, g_target);
    int* xr = resid_norm(out_g);
    EngPhase gu = gemm(eng_plan(m->p_gu, m->q_gu), w.pk_gu, ENG_B_XN, xr, d / TILE_M);
    // two gate/up tiles per item when one each would leave CTAs with two items
    const int asub = gu.T > m->num_sms ? 2 : 1;
    EngPhase& act = row(ENG_ACT, (gu.T + asub - 1) / asub, gu);
    act.sub = asub;
    act.T = gu.T;
    act.out = s->h;
    act.out_ld = F;
    int* h_ready = act.ready;
    const int h_items = act.G;
    EngPhase dn = gemm(eng_plan(m->p_down, m->q_down), w.pk_down, ENG_B_H, h_ready, h_items);
    xn_ready = resid_norm(dn);
  }
  EngPhase hd = gemm(eng_plan(m->p_head, m->q_head), m->pk_head, ENG_B_XN, xn_ready, d / TILE_M);
  EngPhase& lg = row(ENG_LOGITS, V / TILE_M, hd);
  lg.ready = nullptr;
  segs->push_back({seg0, (int)ph.size(), -1, nullptr});
  *ncnt = k + 1;  // + the abort flag
}

static int build_engine(evs_state* s) {
  s->engine_ok = false;
  s->use_engine = false;
  if (!engine_eligible(s->m)) return EVS_OK;
  std::vector<EngPhase> prog;
  std::vector<evs_state::EngSeg> segs;
  size_t ncnt = 0;
  int rf = 0;
  engine_program(s, nullptr, &prog, &segs, &ncnt, &rf);
  void* cnt = nullptr;
  EVS_TRY(dmalloc(s, &cnt, sizeof(int) * ncnt));
  engine_program(s, static_cast<int*>(cnt), &prog, &segs, &ncnt, &rf);
  if (engine_smem(rf) > 232448) return EVS_OK;
  void* dprog = nullptr;
  EVS_TRY(dmalloc(s, &dprog, sizeof(EngPhase) * prog.size()));
  CUDA_TRY(cudaMemcpy(dprog, prog.data(), sizeof(EngPhase) * prog.size(), cudaMemcpyHostToDevice));
  s->eng_prog = static_cast<EngPhase*>(dprog);
  s->eng_segs = segs;
  s->eng_cnt = static_cast<int*>(cnt);
  s->eng_cnt_bytes = sizeof(int) * ncnt;
  s->eng_row_floats = rf;
  s->engine_ok = true;
  s->use_engine = false;  // opt-in: measured slower than the separate kernels (see evs_state_use_engine)
  return EVS_OK;
}

// One verify of a single sequence's block through the engine: counters
// cleared, embedding + first norm, then every span as one persistent launch
// with the attention mixers between spans.
static int enqueue_verify_engine(evs_state* s, const int32_t* tokens, int n, float* logits, const LaunchCtx& Lc) {
  const evs_model* m = s->m;
  const evs_config& c = m->cfg;
  CUDA_TRY(cudaMemsetAsync(s->eng_cnt, 0, s->eng_cnt_bytes, Lc.stream));
  const SeqRows sr = one_seq(n);
  CUDA_TRY(launch_embed_norm(LaunchCtx{Lc.stream, false}, c.dtype, m->embed, tokens, sr, c.d_model, c.vocab,
                             c.norm_eps, s->X, s->xn,
                             one_ptr(s->book)));
  const LaunchCtx Le{Lc.stream, false};
  for (const auto& sg : s->eng_segs) {
    EngArgs a{};
    a.prog = s->eng_prog;
    a.ph0 = sg.ph0;
    a.ph1 = sg.ph1;
    a.n = n;
    a.d = c.d_model;
    a.eps = c.norm_eps;
    a.gabort = s->eng_cnt + s->eng_cnt_bytes / sizeof(int) - 1;
    a.book = s->book;
    a.logits = logits;
    a.V = c.vocab;
    a.row_floats = s->eng_row_floats;
    CUDA_TRY(launch_engine(Le, s->m_xn, s->m_g, s->m_h, a, m->num_sms));
    if (sg.attn_layer >= 0) {
      const LayerS& st = s->S[sg.attn_layer];
      AttnSeq as{};
      as.kc.p[0] = st.kc;
      as.vc.p[0] = st.vc;
      as.kmap.p[0] = st.kmap;
      as.vmap.p[0] = st.vmap;
      as.arrivals.p[0] = s->ab.arrivals;
      as.book.p[0] = s->book;
      as.part_o.p[0] = s->ab.part_o;
      as.part_ml.p[0] = s->ab.part_ml;
      MixSrc src{s->fin, 3 * c.d_model, 1, sg.attn_ws, eng_plan(m->p_in, m->q_in).tab, NTOK};
      CUDA_TRY(launch_attention(Lc, c.dtype, src, c.n_heads, c.head_dim, sr, s->ctx_max, c.attn_chunk, as, s->ab,
                                s->g));
    }
  }
  return EVS_OK;
}

// ------------------------------------------------------------------ verify sequence
// One verify pass over the block rows of nseq sequences: rows [row0[b],
// row0[b+1]) belong to states[b].  The weight GEMMs run once over all rows;
// the work buffers (residual, activations, partials) are states[0]'s, the
// recurrent state, caches and bookkeeping each sequence's own.
int enqueue_verify(evs_state* const* states, const SeqRows& sr, const int32_t* tokens, float* logits,
                   const LaunchCtx& Lc, float* trace = nullptr) {
  evs_state* s = states[0];
  const int n = sr.row0[sr.nseq];
  evs_model* m = s->m;
  const evs_config& c = m->cfg;
  const int d = c.d_model, F = c.d_ffn, V = c.vocab, dt = c.dtype;
  const float eps = c.norm_eps;
  int wsi = 0;
  // Weight matrices in the order the step reads them; each GEMM prefetches
  // the start of the next one into L2 (the head's successor is the next
  // round's first in-projection).
  const int nl = (int)m->L.size();
  auto seq = [&](int k, const Partials** P, const CUtensorMap** map, const uint8_t** pk) {
    k %= 4 * nl + 1;
    if (k == 4 * nl) {
      *P = &m->p_head;
      *map = &m->m_head;
      *pk = m->pk_head;
      return;
    }
    const LayerW& w = m->L[k / 4];
    const Partials* plans[4] = {&m->p_in, &m->p_out, &m->p_gu, &m->p_down};
    const CUtensorMap* maps[4] = {&w.m_in, &w.m_out, &w.m_gu, &w.m_down};
    const uint8_t* pks[4] = {w.pk_in, w.pk_out, w.pk_gu, w.pk_down};
    *P = plans[k % 4];
    *map = maps[k % 4];
    *pk = pks[k % 4];
  };
  int gk = 0;
  // GEMM_FINAL writes fin[tok][col] (row stride ld); GEMM_RESID adds into X
  // and leaves per-tile sums of squares for the next RMSNorm
  const int nt = (n + NTOK - 1) / NTOK;
  // with out set, a stream-K launch leaves its slots (GEMM_SLOTS) instead of
  // running `mode`; *out then says where the consumer reads the result
  // (the slots, or fin for GEMM_FINAL)
  auto gemm = [&](const Partials& plan, const CUtensorMap& wm, const uint8_t* pk, const void* W,
                  const CUtensorMap& xm, const void* Xin, int K, int mode, float* fin, int ld,
                  int bsrc = GEMM_B_TMA, MixSrc* out = nullptr, int cnt_max = SLOTS_MIX_MAX) -> int {
    Partials P = plan;
    if (nt > 1) {
      // more than 16 rows: the stream-K twin, with a ring that fits nt
      // activation tiles per stage
      const Partials* one[5] = {&m->p_in, &m->p_out, &m->p_gu, &m->p_down, &m->p_head};
      const Partials* many[5] = {&m->q_in, &m->q_out, &m->q_gu, &m->q_down, &m->q_head};
      for (int k = 0; k < 5; ++k)
        if (&plan == one[k]) P = *many[k];
      if (P.cl != 0 || bsrc != GEMM_B_TMA || !m->tc)
        return fail(EVS_ERR_UNSUPPORTED, "passes of more than %d rows need the bf16 path without EVS_OPT_NORM_IN_GEMM", NTOK);
      P.stages = std::min(P.stages, gemm_stages_for(0, GEMM_B_TMA, nt));
    }
    P.nt = nt;
    if (out && P.cl == 0 && m->slots && P.max_cnt <= cnt_max) mode = GEMM_SLOTS;
    P.wpk = pk;
    P.bsrc = bsrc;
    P.Kdim = K;
    P.ss_in = s->ss;
    P.ss_tiles = (d + TILE_M - 1) / TILE_M;
    P.norm_d = d;
    P.eps = eps;
    P.hout = static_cast<bf16*>(s->h);
    P.h_cols = F;
    P.ws = s->ws[(wsi++) & 1];
    P.cnt = s->cnt;
    P.mode = mode;
    P.n = n;
    P.fin = fin;
    P.fin_ld = ld;
    P.X = s->X;
    P.ss = s->ss;
    const Partials* np;
    const CUtensorMap* nmap;
    const uint8_t* npk;
    seq(++gk, &np, &nmap, &npk);
    P.nwpk = npk;
    P.pf_units = s->pf_units;
    P.nG = np->G;
    P.nKB = np->KB;
    P.nU = np->U;
    P.ncl = np->cl;
    if (out) {
      *out = MixSrc{fin, ld, 1};
      if (mode == GEMM_SLOTS) {
        out->ws = P.ws;
        out->tab = P.tab;
        out->slot_rows = NTOK * nt;
      }
    }
    if (m->tc)
      CUDA_TRY(launch_gemm_tc(Lc, wm, xm, *nmap, P, K, &s->book->status));
    else
      CUDA_TRY(launch_gemm_simt(Lc, dt, W, Xin, K, P, K));
    return EVS_OK;
  };
  const size_t xbytes = sizeof(float) * (size_t)n * d;
  const int nseq = sr.nseq;
  SeqPtrs<evs_book*> books{};
  SeqPtrs<const evs_book*> cbooks{};
  for (int b = 0; b < nseq; ++b) {
    books.p[b] = states[b]->book;
    cbooks.p[b] = states[b]->book;
  }
  // The first kernel of a verify waits for all earlier work (no programmatic
  // overlap): later kernels read the committed state (lengths, banks, cache
  // rows) before their own dependency wait.
  CUDA_TRY(launch_embed_norm(LaunchCtx{Lc.stream, false}, dt, m->embed, tokens, sr, d, V, eps, s->X, s->xn, books));
  if (trace) CUDA_TRY(cudaMemcpyAsync(trace, s->X, xbytes, cudaMemcpyDeviceToDevice, Lc.stream));
  const bool fz = m->fuse, sg = m->swiglu;
  for (size_t i = 0; i < m->L.size(); ++i) {
    const LayerW& w = m->L[i];
    LayerS& st = s->S[i];
    // the first in-projection reads the embedding kernel's normalised rows;
    // later ones normalise the residual stream themselves when fused
    MixSrc src{};
    if (fz && i > 0)
      EVS_TRY(gemm(m->p_in, w.m_in, w.pk_in, w.w_in, s->m_xf, s->X, d, GEMM_FINAL, s->fin, 3 * d, GEMM_B_NORM, &src));
    else
      EVS_TRY(gemm(m->p_in, w.m_in, w.pk_in, w.w_in, s->m_xn, s->xn, d, GEMM_FINAL, s->fin, 3 * d, GEMM_B_TMA, &src));
    (void)st;
    if (w.kind == EVS_LAYER_FIR) {
      SeqPtrs<float*> rings{};
      for (int b = 0; b < nseq; ++b) rings.p[b] = states[b]->S[i].ring;
      CUDA_TRY(launch_fir(Lc, dt, src, d, sr, w.param, w.param - 1 + m->n_max, w.taps, rings, cbooks, s->g));
    } else if (w.kind == EVS_LAYER_IIR) {
      SeqPtrs<float*> s0{}, s1{};
      for (int b = 0; b < nseq; ++b) s0.p[b] = states[b]->S[i].st[0], s1.p[b] = states[b]->S[i].st[1];
      CUDA_TRY(launch_iir(Lc, dt, src, d, sr, w.param, w.lam, w.res, s0, s1, cbooks, s->g));
    } else {
      AttnSeq as{};
      for (int b = 0; b < nseq; ++b) {
        as.kc.p[b] = states[b]->S[i].kc;
        as.vc.p[b] = states[b]->S[i].vc;
        as.kmap.p[b] = states[b]->S[i].kmap;
        as.vmap.p[b] = states[b]->S[i].vmap;
        as.arrivals.p[b] = states[b]->ab.arrivals;
        as.book.p[b] = states[b]->book;
        as.part_o.p[b] = states[b]->ab.part_o;
        as.part_ml.p[b] = states[b]->ab.part_ml;
      }
      CUDA_TRY(launch_attention(Lc, dt, src, c.n_heads, c.head_dim, sr, s->ctx_max, c.attn_chunk, as, s->ab, s->g));
    }
    // residual GEMM, then (unfused) the RMSNorm of the updated rows: by
    // resid_norm from the GEMM's slots, or by norm_apply after the GEMM's
    // own residual epilogue
    auto resid_gemm = [&](const Partials& plan, const CUtensorMap& wm, const uint8_t* pk, const void* W,
                          const CUtensorMap& xm, const void* Xin, int K) -> int {
      MixSrc rs{};
      EVS_TRY(gemm(plan, wm, pk, W, xm, Xin, K, GEMM_RESID, nullptr, 0, GEMM_B_TMA,
                   fz || !m->slots_resid ? nullptr : &rs, SLOTS_RESID_MAX));
      if (fz) return EVS_OK;
      if (rs.ws)
        CUDA_TRY(launch_resid_norm(Lc, dt, s->X, rs, n, d, eps, s->xn));
      else
        CUDA_TRY(launch_norm_apply(Lc, dt, s->X, s->ss, n, d, eps, s->xn));
      return EVS_OK;
    };
    EVS_TRY(resid_gemm(m->p_out, w.m_out, w.pk_out, w.w_out, s->m_g, s->g, d));
    const int gu_mode = sg ? GEMM_SWIGLU : GEMM_FINAL;
    MixSrc gsrc{};
    EVS_TRY(gemm(m->p_gu, w.m_gu, w.pk_gu, w.w_gu, fz ? s->m_xf : s->m_xn, fz ? (const void*)s->X : s->xn, d, gu_mode,
                 s->fin, 2 * F, fz ? GEMM_B_NORM : GEMM_B_TMA, sg ? nullptr : &gsrc));
    if (!sg) CUDA_TRY(launch_mlp_act(Lc, dt, gsrc, n, F, m->packed, s->h));
    EVS_TRY(resid_gemm(m->p_down, w.m_down, w.pk_down, w.w_down, s->m_h, s->h, F));
    if (trace)
      CUDA_TRY(cudaMemcpyAsync(trace + (i + 1) * (size_t)n * d, s->X, xbytes, cudaMemcpyDeviceToDevice, Lc.stream));
  }
  if (fz)
    EVS_TRY(gemm(m->p_head, m->m_head, m->pk_head, m->head, s->m_xf, s->X, d, GEMM_FINAL, logits, V, GEMM_B_NORM));
  else
    EVS_TRY(gemm(m->p_head, m->m_head, m->pk_head, m->head, s->m_xn, s->xn, d, GEMM_FINAL, logits, V));
  return EVS_OK;
}

int enqueue_verify(evs_state* s, const int32_t* tokens, int n, float* logits, const LaunchCtx& Lc,
                   float* trace = nullptr) {
  if (s->use_engine && !trace) return enqueue_verify_engine(s, tokens, n, logits, Lc);
  return enqueue_verify(&s, one_seq(n), tokens, logits, Lc, trace);
}

struct RoundArgs {
  float* p;
  const float* q;
  const int32_t* drafts;  // = tokens + 1
  const float* u;
  float T;
  int top_k, mode;
  int32_t *acc, *otok;
};

int enqueue_round(evs_state* s, const int32_t* tokens, int n, float* logits, const RoundArgs& r,
                  const LaunchCtx& Lc) {
  EVS_TRY(enqueue_verify(s, tokens, n, logits, Lc));
  const int V = s->m->cfg.vocab;
  const float* P = logits;
  if (r.mode == EVS_SAMPLE) {
    CUDA_TRY(launch_probs(Lc, logits, n, V, r.T, r.top_k, r.p));
    P = r.p;
  }
  CUDA_TRY(launch_accept(Lc, P, r.q, r.drafts, r.u, n, V, r.mode, r.acc, r.otok, s->book, true));
  return EVS_OK;
}

// Batched round: one verify pass over every sequence's block, then (sample
// mode) the target distributions of all rows, the accept rule per sequence
// (one CTA each) and every sequence's commit with keep = accepted + 1.
int enqueue_round_batch(evs_state* const* states, const SeqRows& sr, const int32_t* tokens, float* logits,
                        const RoundArgs& r, const LaunchCtx& Lc) {
  EVS_TRY(enqueue_verify(states, sr, tokens, logits, Lc));
  const int V = states[0]->m->cfg.vocab;
  const float* P = logits;
  if (r.mode == EVS_SAMPLE) {
    CUDA_TRY(launch_probs(Lc, logits, sr.row0[sr.nseq], V, r.T, r.top_k, r.p));
    P = r.p;
  }
  SeqPtrs<evs_book*> books{};
  for (int b = 0; b < sr.nseq; ++b) books.p[b] = states[b]->book;
  CUDA_TRY(launch_accept_batch(Lc, P, r.q, r.drafts, r.u, sr, V, r.mode, r.acc, r.otok, books, true));
  return EVS_OK;
}

GraphEntry* find_graph(evs_state* s, const GraphEntry& key) {
  for (auto& g : s->graphs)
    if (g.round == key.round && g.n == key.n && g.tok == key.tok && g.logits == key.logits &&
        g.mode == key.mode && g.top_k == key.top_k && g.T == key.T && g.p == key.p && g.q == key.q &&
        g.u == key.u && g.acc == key.acc && g.otok == key.otok && g.nseq == key.nseq && g.host_io == key.host_io &&
        std::equal(g.uid, g.uid + g.nseq, key.uid) && std::equal(g.ns, g.ns + g.nseq, key.ns))
      return &g;
  return nullptr;
}

template <typename F>
int run_captured(evs_state* s, GraphEntry key, cudaStream_t stream, F&& body) {
  if (!s->use_graphs) {
    LaunchCtx Lc{stream, s->pdl};
    return body(Lc);
  }
  GraphEntry* g = find_graph(s, key);
  if (!g) {
    if (s->graphs.size() >= 16) {  // evict the least recently used
      size_t victim = 0;
      for (size_t i = 1; i < s->graphs.size(); ++i)
        if (s->graphs[i].last_use < s->graphs[victim].last_use) victim = i;
      cudaGraphExecDestroy(s->graphs[victim].exec);
      s->graphs.erase(s->graphs.begin() + victim);
    }
    const long long before = g_launches.load();
    CUDA_TRY(cudaStreamBeginCapture(s->cap, cudaStreamCaptureModeRelaxed));
    LaunchCtx Lc{s->cap, s->pdl};
    int r = body(Lc);
    cudaGraph_t graph = nullptr;
    cudaError_t e = cudaStreamEndCapture(s->cap, &graph);
    if (r != EVS_OK) {
      if (graph) cudaGraphDestroy(graph);
      return r;
    }
    if (e != cudaSuccess) return fail(EVS_ERR_CUDA, "stream capture failed: %s", cudaGetErrorString(e));
    cudaGraphExec_t exec = nullptr;
    e = cudaGraphInstantiate(&exec, graph, 0);
    cudaGraphDestroy(graph);
    if (e != cudaSuccess) return fail(EVS_ERR_CUDA, "graph instantiate failed: %s", cudaGetErrorString(e));
    key.exec = exec;
    key.kernels = (int)(g_launches.load() - before);
    g_launches -= key.kernels;  // counted again at each launch
    s->graphs.push_back(key);
    g = &s->graphs.back();
  }
  g->last_use = ++s->tick;
  CUDA_TRY(cudaGraphLaunch(g->exec, stream));
  count_launch(g->kernels);
  return EVS_OK;
}

int check_cfg(const evs_config* c) {
  if (!c) return fail(EVS_ERR_ARG, "null config");
  if (c->vocab <= 0 || c->d_model <= 0 || c->n_layers <= 0 || c->d_ffn <= 0)
    return fail(EVS_ERR_ARG, "vocab, d_model, n_layers, d_ffn must be positive");
  if (c->gamma_max < 0 || c->gamma_max + 1 > NTOK) return fail(EVS_ERR_ARG, "gamma_max must be in [0, %d]", NTOK - 1);
  if (c->dtype != EVS_BF16 && c->dtype != EVS_F32) return fail(EVS_ERR_ARG, "dtype must be EVS_BF16 or EVS_F32");
  if (!c->layer_kind_host || !c->layer_param_host) return fail(EVS_ERR_ARG, "null layer arrays");
  if (c->d_model % 32) return fail(EVS_ERR_UNSUPPORTED, "d_model must be a multiple of 32");
  if (!(c->norm_eps >= 0.f)) return fail(EVS_ERR_ARG, "norm_eps must be >= 0");
  if (c->dtype == EVS_BF16) {
    if (c->d_model % 128 || (2 * c->d_ffn) % 128 || c->vocab % 128 || c->d_ffn % 64)
      return fail(EVS_ERR_UNSUPPORTED, "bf16 path needs d_model, 2*d_ffn, vocab multiples of 128 and d_ffn of 64");
  }
  for (int i = 0; i < c->n_layers; ++i) {
    const int k = c->layer_kind_host[i], p = c->layer_param_host[i];
    if (k == EVS_LAYER_FIR) {
      if (p < 1 || p > 256) return fail(EVS_ERR_UNSUPPORTED, "layer %d: FIR length must be in [1, 256]", i);
    } else if (k == EVS_LAYER_IIR) {
      if (p < 1 || p > 32 || (p & (p - 1))) return fail(EVS_ERR_UNSUPPORTED, "layer %d: IIR poles must be a power of two <= 32", i);
      if (c->d_model % (256 / p)) return fail(EVS_ERR_UNSUPPORTED, "layer %d: d_model * poles must be a multiple of 256", i);
    } else if (k == EVS_LAYER_ATTN) {
      if (c->n_heads * c->head_dim != c->d_model) return fail(EVS_ERR_ARG, "n_heads * head_dim != d_model");
      if (c->head_dim != 32 && c->head_dim != 64 && c->head_dim != 128)
        return fail(EVS_ERR_UNSUPPORTED, "head_dim must be 32, 64 or 128");
      if (c->attn_chunk != 32 && c->attn_chunk != 64 && c->attn_chunk != 128 && c->attn_chunk != 256)
        return fail(EVS_ERR_UNSUPPORTED, "attn_chunk must be 32, 64, 128 or 256");
      if (!(c->rope_base > 0.f)) return fail(EVS_ERR_ARG, "rope_base must be > 0");
    } else {
      return fail(EVS_ERR_ARG, "layer %d: unknown kind %d", i, k);
    }
  }
  return EVS_OK;
}

}  // namespace

// =================================================================== model
extern "C" int evs_model_create(const evs_config* cfg, const evs_weights* w, evs_model** out) {
  if (!out) return fail(EVS_ERR_ARG, "null out");
  *out = nullptr;
  EVS_TRY(check_cfg(cfg));
  if (!w || !w->embed || !w->lm_head || !w->layers_host) return fail(EVS_ERR_ARG, "null weights");
  evs_model* m = new evs_model();
  m->cfg = *cfg;
  m->kind.assign(cfg->layer_kind_host, cfg->layer_kind_host + cfg->n_layers);
  m->param.assign(cfg->layer_param_host, cfg->layer_param_host + cfg->n_layers);
  m->cfg.layer_kind_host = m->kind.data();
  m->cfg.layer_param_host = m->param.data();
  int r = num_sms_current(&m->num_sms);
  if (r != EVS_OK) {
    delete m;
    return r;
  }
  m->tc = cfg->dtype == EVS_BF16;
  m->embed = w->embed;
  m->head = w->lm_head;
  m->n_max = cfg->gamma_max + 1;
  m->has_attn = false;
  {
    const int opt = cfg->options;
    m->packed = m->tc && cfg->d_ffn % (TILE_M / 2) == 0;
    m->swiglu = m->packed && (opt & EVS_OPT_SWIGLU_EPILOGUE);
    // fp32 rows staged by TMA need 16-byte row strides
    m->fuse = m->packed && cfg->d_model % 4 == 0 && (opt & EVS_OPT_NORM_IN_GEMM);
    m->slots = m->tc && !(opt & EVS_OPT_GEMM_SUMS_SLOTS);
    m->slots_resid = m->slots && resid_norm_ok(cfg->d_model);
  }
  const int d = cfg->d_model, F = cfg->d_ffn, V = cfg->vocab;
  char err[256] = {0};
  auto enc = [&](CUtensorMap* map, const void* base, int N, int K) -> bool {
    if (!m->tc) return true;
    if (!aligned16(base)) {
      snprintf(err, sizeof err, "weight pointer not 16-byte aligned");
      return false;
    }
    return encode_tmap_2d(map, base, (uint64_t)K, (uint64_t)N, TILE_K, TILE_M, err, sizeof err);
  };
  for (int i = 0; i < cfg->n_layers; ++i) {
    const evs_layer_weights& lw = w->layers_host[i];
    LayerW L{};
    L.kind = m->kind[i];
    L.param = m->param[i];
    L.w_in = lw.w_in;
    L.w_out = lw.w_out;
    L.w_gu = lw.w_gu;
    L.w_down = lw.w_down;
    L.taps = lw.fir_taps;
    L.lam = lw.iir_lambda;
    L.res = lw.iir_residue;
    if (!L.w_in || !L.w_out || !L.w_gu || !L.w_down ||
        (L.kind == EVS_LAYER_FIR && !L.taps) || (L.kind == EVS_LAYER_IIR && (!L.lam || !L.res))) {
      delete m;
      return fail(EVS_ERR_ARG, "layer %d: null weight pointer", i);
    }
    if (L.kind == EVS_LAYER_ATTN) m->has_attn = true;
    if (!enc(&L.m_in, L.w_in, 3 * d, d) || !enc(&L.m_out, L.w_out, d, d) || !enc(&L.m_gu, L.w_gu, 2 * F, d) ||
        !enc(&L.m_down, L.w_down, d, F)) {
      delete m;
      return fail(EVS_ERR_CUDA, "layer %d: %s", i, err);
    }
    m->L.push_back(L);
  }
  if (!enc(&m->m_head, m->head, V, d)) {
    delete m;
    return fail(EVS_ERR_CUDA, "head: %s", err);
  }
  {
    std::vector<GemmPlan> plans(10);
    const int shapes[5][2] = {{3 * d, d}, {d, d}, {2 * F, d}, {d, F}, {V, d}};
    Partials* dst[10] = {&m->p_in, &m->p_out, &m->p_gu, &m->p_down, &m->p_head,
                         &m->q_in, &m->q_out, &m->q_gu, &m->q_down, &m->q_head};
    size_t tb = 0;
    m->ws_bytes = 0;
    for (int k = 0; k < 5; ++k) {
      const bool allow_cl = m->tc;
      const bool resid = k == 1 || k == 3;
      const int cl = allow_cl && !(resid && m->slots_resid) ? gemm_cluster_choice(shapes[k][0], shapes[k][1], m->num_sms)
                                                            : 0;
      const bool planned = cl ? plan_gemm_cluster(shapes[k][0], shapes[k][1], cl, &plans[k])
                              : plan_gemm(shapes[k][0], shapes[k][1], m->num_sms, &plans[k]);
      if (!planned) {
        delete m;
        return fail(EVS_ERR_UNSUPPORTED, "GEMM shape %d x %d has too many column tiles", shapes[k][0], shapes[k][1]);
      }
      // ring depth that fits next to this GEMM's B-source staging
      const int bs[5] = {GEMM_B_NORM, GEMM_B_TMA, GEMM_B_NORM, GEMM_B_TMA, GEMM_B_NORM};
      if (m->tc)
        plans[k].P.stages =
            std::min(plans[k].P.stages, gemm_stages_for(plans[k].P.cl, m->fuse ? bs[k] : GEMM_B_TMA));
      // stream-K twin over the same CTA unit ranges (G = T * cl for a
      // cluster plan), for passes of more than NTOK rows
      GemmPlan& q = plans[5 + k];
      if (!plan_gemm_grid(shapes[k][0], shapes[k][1], plans[k].P.G, &q)) {
        delete m;
        return fail(EVS_ERR_UNSUPPORTED, "GEMM shape %d x %d: no stream-K plan", shapes[k][0], shapes[k][1]);
      }
      q.P.stages = plans[k].P.stages;
      tb += table_bytes(plans[k]) + table_bytes(q);
      m->ws_bytes = std::max(m->ws_bytes, partials_bytes(plans[k]));
      if (m->tc) m->ws_bytes = std::max(m->ws_bytes, partials_bytes(q, ROWS_MAX));
    }
    cudaError_t e = cudaMalloc(&m->tab_dev, tb);
    if (e != cudaSuccess) {
      delete m;
      return fail(EVS_ERR_OOM, "cudaMalloc(slot tables): %s", cudaGetErrorString(e));
    }
    size_t off = 0;
    for (int k = 0; k < 10; ++k) {
      const int T = (int)(table_bytes(plans[k]) / sizeof(int4));
      e = cudaMemcpy(m->tab_dev + off, plans[k].tab, table_bytes(plans[k]), cudaMemcpyHostToDevice);
      if (e != cudaSuccess) {
        cudaFree(m->tab_dev);
        delete m;
        return fail(EVS_ERR_CUDA, "upload slot tables: %s", cudaGetErrorString(e));
      }
      *dst[k] = plans[k].P;
      dst[k]->tab = m->tab_dev + off;
      off += T;
    }
  }
  // bf16: repack every projection matrix into the unit-major swizzled layout
  // the tensor-core GEMM streams with contiguous bulk copies
  if (m->packed) {
    const size_t per_layer = packed_bytes(m->p_in) + packed_bytes(m->p_out) + packed_bytes(m->p_gu) +
                             packed_bytes(m->p_down);
    const size_t total = per_layer * m->L.size() + packed_bytes(m->p_head);
    cudaError_t e = cudaMalloc(&m->wpack, total);
    if (e != cudaSuccess) {
      cudaGetLastError();
      m->wpack = nullptr;
      evs_model_destroy(m);
      return fail(EVS_ERR_OOM, "cudaMalloc(%zu) for packed weights: %s", total, cudaGetErrorString(e));
    }
    size_t off = 0;
    auto pack = [&](const void* W, int N, int K, const Partials& P, int swg_half = 0) -> const uint8_t* {
      uint8_t* dst = m->wpack + off;
      off += packed_bytes(P);
      if (e == cudaSuccess) e = launch_pack_weights(0, static_cast<const bf16*>(W), N, K, P, swg_half, dst);
      return dst;
    };
    for (LayerW& L : m->L) {
      L.pk_in = pack(L.w_in, 3 * d, d, m->p_in);
      L.pk_out = pack(L.w_out, d, d, m->p_out);
      L.pk_gu = pack(L.w_gu, 2 * F, d, m->p_gu, F);  // gate/up interleaved by 64 rows
      L.pk_down = pack(L.w_down, d, F, m->p_down);
    }
    m->pk_head = pack(m->head, V, d, m->p_head);
    if (e == cudaSuccess) e = cudaStreamSynchronize(0);
    if (e != cudaSuccess) {
      evs_model_destroy(m);
      return fail(EVS_ERR_CUDA, "packing weights: %s", cudaGetErrorString(e));
    }
  }
  *out = m;
  return EVS_OK;
}

extern "C" int evs_model_destroy(evs_model* m) {
  if (m && m->tab_dev) cudaFree(m->tab_dev);
  if (m && m->wpack) cudaFree(m->wpack);
  delete m;
  return EVS_OK;
}

// =================================================================== state
static void state_free(evs_state* s) {
  if (!s) return;
  for (auto& g : s->graphs) cudaGraphExecDestroy(g.exec);
  if (s->cap) cudaStreamDestroy(s->cap);
  for (void* p : s->allocs) cudaFree(p);
  if (s->io_pinned) cudaFreeHost(s->io_pinned);
  delete s;
}

static evs_book initial_book() {
  evs_book b{};
  b.iir_slot = -1;
  return b;
}

extern "C" int evs_state_create(evs_model* m, int64_t ctx_max, evs_state** out) {
  if (!m || !out) return fail(EVS_ERR_ARG, "null argument");
  if (ctx_max < 1 || ctx_max > (1ll << 30)) return fail(EVS_ERR_ARG, "ctx_max out of range");
  *out = nullptr;
  evs_state* s = new evs_state();
  s->m = m;
  s->uid = ++g_state_uid;
  s->ctx_max = ctx_max;
  s->use_graphs = true;
  s->pdl = true;
  // 4 units (64 KB) per CTA, 9.7 MB in all: measured best on the 7B-shaped
  // step (deeper prefetches compete with the running GEMM's own stream)
  s->pf_units = 4;
  const evs_config& c = m->cfg;
  const int d = c.d_model, F = c.d_ffn, nm = m->n_max;
  const size_t es = esize(c.dtype);
  int r = EVS_OK;
#define ALLOC(ptr, bytes)                                              \
  do {                                                                 \
    void* p_ = nullptr;                                                \
    r = dmalloc(s, &p_, (bytes));                                      \
    if (r != EVS_OK) { state_free(s); return r; }                      \
    ptr = reinterpret_cast<decltype(ptr)>(p_);                         \
  } while (0)
  ALLOC(s->book, sizeof(evs_book));
  const size_t R = ROWS_MAX;
  ALLOC(s->X, sizeof(float) * R * d);
  ALLOC(s->xn, es * R * d);
  ALLOC(s->g, es * R * d);
  ALLOC(s->h, es * R * F);
  ALLOC(s->fin, sizeof(float) * R * std::max(3 * d, std::max(2 * F, c.vocab)));
  ALLOC(s->pout, sizeof(float) * NTOK * std::max(3 * d, std::max(2 * F, c.vocab)));
  ALLOC(s->ss, sizeof(float) * R * ((d + TILE_M - 1) / TILE_M));
  s->cnt_len = (std::max(3 * d, std::max(2 * F, c.vocab)) + TILE_M - 1) / TILE_M;
  ALLOC(s->cnt, sizeof(int) * s->cnt_len);
  ALLOC(s->io_dev, sizeof(int32_t) * (NTOK + 2));
  {
    void* ph = nullptr;
    cudaError_t e = cudaHostAlloc(&ph, sizeof(int32_t) * (NTOK + 2), cudaHostAllocDefault);
    if (e != cudaSuccess) {
      cudaGetLastError();
      state_free(s);
      return fail(EVS_ERR_OOM, "cudaHostAlloc(staging) failed: %s", cudaGetErrorString(e));
    }
    s->io_pinned = static_cast<int32_t*>(ph);
  }
  size_t wsb = 0;
  wsb = m->ws_bytes;
  ALLOC(s->ws[0], wsb);
  ALLOC(s->ws[1], wsb);
  if (m->has_attn) {
    const size_t ab = attn_scratch_bytes(c.n_heads, c.head_dim, ctx_max, c.attn_chunk);
    ALLOC(s->attn_scratch, ab);
    attn_bufs_from_scratch(s->attn_scratch, c.n_heads, c.head_dim, ctx_max, c.attn_chunk, &s->ab);
    cudaError_t e = fill_rope_table(s->ab, c.head_dim, c.rope_base, 0);
    if (e != cudaSuccess) {
      state_free(s);
      return fail(EVS_ERR_CUDA, "rotary table: %s", cudaGetErrorString(e));
    }
  }
  s->S.resize(m->L.size());
  for (size_t i = 0; i < m->L.size(); ++i) {
    LayerS& st = s->S[i];
    st = LayerS{};
    const LayerW& L = m->L[i];
    if (L.kind == EVS_LAYER_FIR) {
      ALLOC(st.ring, sizeof(float) * (size_t)(L.param - 1 + nm) * d);
    } else if (L.kind == EVS_LAYER_IIR) {
      for (int b = 0; b < 2; ++b) ALLOC(st.st[b], sizeof(float) * 2 * (size_t)nm * d * L.param);
    } else {
      ALLOC(st.kc, es * (size_t)c.n_heads * ctx_max * c.head_dim);
      ALLOC(st.vc, es * (size_t)c.n_heads * ctx_max * c.head_dim);
    }
  }
  if (m->has_attn && attn_tma_eligible(c.dtype, c.n_heads, c.head_dim, ctx_max)) {
    // tensor maps of every attention cache, encoded once (the caches never move)
    std::vector<CUtensorMap> maps;
    char err[256] = {0};
    for (const LayerS& st : s->S) {
      if (!st.kc) continue;
      CUtensorMap km, vm;
      if (!encode_kv_maps(&km, &vm, st.kc, st.vc, c.n_heads, c.head_dim, ctx_max, err, sizeof err)) {
        state_free(s);
        return fail(EVS_ERR_CUDA, "KV tensor map: %s", err);
      }
      maps.push_back(km);
      maps.push_back(vm);
    }
    CUtensorMap* dmaps = nullptr;
    ALLOC(dmaps, sizeof(CUtensorMap) * maps.size());
    cudaError_t e = cudaMemcpy(dmaps, maps.data(), sizeof(CUtensorMap) * maps.size(), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) {
      state_free(s);
      return fail(EVS_ERR_CUDA, "KV tensor map upload: %s", cudaGetErrorString(e));
    }
    int j = 0;
    for (LayerS& st : s->S) {
      if (!st.kc) continue;
      st.kmap = dmaps + 2 * j;
      st.vmap = dmaps + 2 * j + 1;
      ++j;
    }
  }
#undef ALLOC
  if (m->tc) {
    char err[256] = {0};
    if (!encode_tmap_2d(&s->m_xn, s->xn, d, ROWS_MAX, TILE_K, NTOK, err, sizeof err) ||
        !encode_tmap_2d(&s->m_g, s->g, d, ROWS_MAX, TILE_K, NTOK, err, sizeof err) ||
        !encode_tmap_2d(&s->m_h, s->h, F, ROWS_MAX, TILE_K, NTOK, err, sizeof err) ||
        (m->fuse && !encode_tmap_2d_f32(&s->m_xf, s->X, d, ROWS_MAX, TILE_K, NTOK, err, sizeof err))) {
      state_free(s);
      return fail(EVS_ERR_CUDA, "activation tensor map: %s", err);
    }
  }
  cudaError_t e = cudaStreamCreateWithFlags(&s->cap, cudaStreamNonBlocking);
  if (e != cudaSuccess) {
    state_free(s);
    return fail(EVS_ERR_CUDA, "cudaStreamCreate: %s", cudaGetErrorString(e));
  }
  // zero activations once (rows beyond a block's n are read but never used)
  cudaMemset(s->xn, 0, es * R * d);
  cudaMemset(s->g, 0, es * R * d);
  cudaMemset(s->h, 0, es * R * F);
  r = evs_state_reset(s, 0);
  if (r == EVS_OK) r = build_engine(s);
  if (r == EVS_OK) {
    e = cudaDeviceSynchronize();
    if (e != cudaSuccess) r = fail(EVS_ERR_CUDA, "state init: %s", cudaGetErrorString(e));
  }
  if (r != EVS_OK) {
    state_free(s);
    return r;
  }
  *out = s;
  return EVS_OK;
}

extern "C" int evs_state_destroy(evs_state* s) {
  if (s) cudaDeviceSynchronize();
  state_free(s);
  return EVS_OK;
}

extern "C" int evs_state_reset(evs_state* s, cudaStream_t stream) {
  if (!s) return fail(EVS_ERR_ARG, "null state");
  const evs_model* m = s->m;
  for (size_t i = 0; i < m->L.size(); ++i) {
    const LayerW& L = m->L[i];
    if (L.kind == EVS_LAYER_FIR)  // positions before 0 read as zero inputs
      CUDA_TRY(cudaMemsetAsync(s->S[i].ring, 0, sizeof(float) * (size_t)(L.param - 1 + m->n_max) * m->cfg.d_model,
                               stream));
  }
  LaunchCtx Lc{stream, false};
  CUDA_TRY(cudaMemsetAsync(s->cnt, 0, sizeof(int) * s->cnt_len, stream));
  if (s->m->has_attn) CUDA_TRY(cudaMemsetAsync(s->ab.arrivals, 0, sizeof(int) * s->m->cfg.n_heads, stream));
  CUDA_TRY(launch_book_set(Lc, s->book, initial_book()));
  s->host_pos = 0;
  s->host_pos_known = true;
  s->host_pending = 0;
  return EVS_OK;
}

extern "C" int evs_state_layer_view(const evs_state* s, int32_t layer, evs_layer_view* out) {
  if (!s || !out) return fail(EVS_ERR_ARG, "null argument");
  if (layer < 0 || layer >= (int)s->S.size()) return fail(EVS_ERR_ARG, "layer out of range");
  const LayerS& st = s->S[layer];
  out->kind = s->m->L[layer].kind;
  out->param = s->m->L[layer].param;
  out->fir_ring = st.ring;
  out->reserved = nullptr;
  out->iir_all[0] = st.st[0];
  out->iir_all[1] = st.st[1];
  out->k_cache = st.kc;
  out->v_cache = st.vc;
  out->ctx_max = s->ctx_max;
  out->n_max = s->m->n_max;
  return EVS_OK;
}

extern "C" int evs_state_book_dev(const evs_state* s, evs_book** out) {
  if (!s || !out) return fail(EVS_ERR_ARG, "null argument");
  *out = s->book;
  return EVS_OK;
}

extern "C" int evs_state_book_read(const evs_state* s, evs_book* out, cudaStream_t stream) {
  if (!s || !out) return fail(EVS_ERR_ARG, "null argument");
  CUDA_TRY(cudaMemcpyAsync(out, s->book, sizeof(evs_book), cudaMemcpyDeviceToHost, stream));
  CUDA_TRY(cudaStreamSynchronize(stream));
  return EVS_OK;
}

extern "C" int evs_state_book_write(evs_state* s, const evs_book* in, cudaStream_t stream) {
  if (!s || !in) return fail(EVS_ERR_ARG, "null argument");
  if (in->pos < 0 || in->pos > s->ctx_max || in->reserved0 || in->reserved1 || (in->iir_bank & ~1) ||
      in->iir_slot < -1 || in->iir_slot >= s->m->n_max ||
      in->pending_n < 0 || in->pending_n > s->m->n_max)
    return fail(EVS_ERR_ARG, "book field out of range");
  LaunchCtx Lc{stream, false};
  CUDA_TRY(launch_book_set(Lc, s->book, *in));
  CUDA_TRY(cudaStreamSynchronize(stream));
  s->host_pos = in->pos;
  s->host_pos_known = true;
  s->host_pending = in->pending_n;
  return EVS_OK;
}

extern "C" int evs_state_check(evs_state* s, cudaStream_t stream, int32_t* status) {
  evs_book b;
  EVS_TRY(evs_state_book_read(s, &b, stream));
  if (status) *status = b.status;
  if (b.status) return fail(EVS_ERR_DEVICE, "device status 0x%x", b.status);
  return EVS_OK;
}

extern "C" int evs_state_use_graphs(evs_state* s, int32_t enable) {
  if (!s) return fail(EVS_ERR_ARG, "null state");
  s->use_graphs = enable != 0;
  return EVS_OK;
}

extern "C" int evs_state_use_engine(evs_state* s, int32_t enable) {
  if (!s) return fail(EVS_ERR_ARG, "null state");
  if (enable && !s->engine_ok) return fail(EVS_ERR_UNSUPPORTED, "the persistent engine does not take this model");
  if ((enable != 0) != s->use_engine) {
    for (auto& g : s->graphs) cudaGraphExecDestroy(g.exec);  // captured with the other path
    s->graphs.clear();
  }
  s->use_engine = enable != 0;
  return EVS_OK;
}

extern "C" int evs_state_snapshot(const evs_state* src, evs_state* dst, cudaStream_t stream) {
  if (!src || !dst) return fail(EVS_ERR_ARG, "null state");
  if (src->m != dst->m || src->ctx_max != dst->ctx_max)
    return fail(EVS_ERR_ARG, "snapshot needs the same model and ctx_max");
  evs_book b;
  EVS_TRY(evs_state_book_read(src, &b, stream));
  const evs_model* m = src->m;
  const evs_config& c = m->cfg;
  for (size_t i = 0; i < m->L.size(); ++i) {
    const LayerW& L = m->L[i];
    const LayerS &a = src->S[i], &z = dst->S[i];
    if (L.kind == EVS_LAYER_FIR) {
      CUDA_TRY(cudaMemcpyAsync(z.ring, a.ring, sizeof(float) * (size_t)(L.param - 1 + m->n_max) * c.d_model,
                               cudaMemcpyDeviceToDevice, stream));
    } else if (L.kind == EVS_LAYER_IIR) {
      for (int k = 0; k < 2; ++k)
        CUDA_TRY(cudaMemcpyAsync(z.st[k], a.st[k], sizeof(float) * 2 * (size_t)m->n_max * c.d_model * L.param,
                                 cudaMemcpyDeviceToDevice, stream));
    }
  }
  CUDA_TRY(cudaMemcpyAsync(dst->book, src->book, sizeof(evs_book), cudaMemcpyDeviceToDevice, stream));
  dst->host_pos = b.pos;
  dst->host_pos_known = true;
  dst->host_pending = b.pending_n;
  return EVS_OK;
}

extern "C" int evs_state_clone(const evs_state* src, evs_state* dst, cudaStream_t stream) {
  if (!src || !dst) return fail(EVS_ERR_ARG, "null state");
  if (src->m != dst->m || src->ctx_max != dst->ctx_max) return fail(EVS_ERR_ARG, "clone needs the same model and ctx_max");
  evs_book b;
  EVS_TRY(evs_state_book_read(src, &b, stream));
  const evs_model* m = src->m;
  const evs_config& c = m->cfg;
  const size_t es = esize(c.dtype);
  for (size_t i = 0; i < m->L.size(); ++i) {
    const LayerW& L = m->L[i];
    const LayerS &a = src->S[i], &z = dst->S[i];
    if (L.kind == EVS_LAYER_FIR) {
      CUDA_TRY(cudaMemcpyAsync(z.ring, a.ring, sizeof(float) * (size_t)(L.param - 1 + m->n_max) * c.d_model,
                               cudaMemcpyDeviceToDevice, stream));
    } else if (L.kind == EVS_LAYER_IIR) {
      for (int k = 0; k < 2; ++k)
        CUDA_TRY(cudaMemcpyAsync(z.st[k], a.st[k], sizeof(float) * 2 * (size_t)m->n_max * c.d_model * L.param,
                                 cudaMemcpyDeviceToDevice, stream));
    } else if (b.pos + b.pending_n > 0) {
      const size_t rowb = es * c.head_dim, pitch = rowb * src->ctx_max;
      const size_t rows = (size_t)std::min<long long>(src->ctx_max, (long long)b.pos + b.pending_n);
      CUDA_TRY(cudaMemcpy2DAsync(z.kc, pitch, a.kc, pitch, rows * rowb, c.n_heads, cudaMemcpyDeviceToDevice, stream));
      CUDA_TRY(cudaMemcpy2DAsync(z.vc, pitch, a.vc, pitch, rows * rowb, c.n_heads, cudaMemcpyDeviceToDevice, stream));
    }
  }
  CUDA_TRY(cudaMemcpyAsync(dst->book, src->book, sizeof(evs_book), cudaMemcpyDeviceToDevice, stream));
  dst->host_pos = b.pos;
  dst->host_pos_known = true;
  dst->host_pending = b.pending_n;
  return EVS_OK;
}

// =================================================================== path
static int check_block(evs_state* s, int n) {
  if (n < 1 || n > s->m->n_max) return fail(EVS_ERR_ARG, "n=%d outside [1, gamma_max+1=%d]", n, s->m->n_max);
  if (s->host_pending) return fail(EVS_ERR_STATE, "a verified block of %d tokens awaits commit", s->host_pending);
  if (s->host_pos_known && (long long)s->host_pos + n > s->ctx_max)
    return fail(EVS_ERR_CAPACITY, "position %d + %d exceeds ctx_max %lld", s->host_pos, n, s->ctx_max);
  return EVS_OK;
}

extern "C" int evs_verify_block(evs_state* s, const int32_t* tokens, int32_t n, float* logits, cudaStream_t stream) {
  if (!s || !tokens || !logits) return fail(EVS_ERR_ARG, "null argument");
  EVS_TRY(check_block(s, n));
  GraphEntry key{};
  key.n = n;
  key.tok = tokens;
  key.logits = logits;
  EVS_TRY(run_captured(s, key, stream, [&](const LaunchCtx& Lc) { return enqueue_verify(s, tokens, n, logits, Lc); }));
  s->host_pending = n;
  return EVS_OK;
}

// Checks a batch (states distinct, one model and ctx_max, each block valid,
// rows within the model's pass limit) and fills its row ranges.
static int check_batch(evs_state* const* states, int32_t nseq, const int32_t* n_host, SeqRows* sr) {
  if (nseq < 1 || nseq > MAX_SEQ) return fail(EVS_ERR_ARG, "nseq=%d outside [1, %d]", nseq, MAX_SEQ);
  *sr = SeqRows{};
  sr->nseq = nseq;
  for (int b = 0; b < nseq; ++b) {
    evs_state* s = states[b];
    if (!s) return fail(EVS_ERR_ARG, "null state %d", b);
    if (s->m != states[0]->m || s->ctx_max != states[0]->ctx_max)
      return fail(EVS_ERR_ARG, "batched states need the same model and ctx_max");
    for (int q = 0; q < b; ++q)
      if (states[q] == s) return fail(EVS_ERR_ARG, "state %d appears twice", b);
    EVS_TRY(check_block(s, n_host[b]));
    sr->row0[b + 1] = sr->row0[b] + n_host[b];
  }
  const evs_model* m = states[0]->m;
  const int rows_max = m->tc && !m->fuse ? ROWS_MAX : NTOK;
  if (sr->row0[nseq] > rows_max)
    return fail(sr->row0[nseq] > ROWS_MAX ? EVS_ERR_ARG : EVS_ERR_UNSUPPORTED,
                "%d block rows in total, at most %d for this model", sr->row0[nseq], rows_max);
  return EVS_OK;
}

extern "C" int evs_verify_batch(evs_state* const* states, int32_t nseq, const int32_t* tokens, const int32_t* n_host,
                                float* logits, cudaStream_t stream) {
  if (!states || !tokens || !n_host || !logits) return fail(EVS_ERR_ARG, "null argument");
  SeqRows sr{};
  EVS_TRY(check_batch(states, nseq, n_host, &sr));
  LaunchCtx Lc{stream, states[0]->pdl};
  EVS_TRY(enqueue_verify(states, sr, tokens, logits, Lc));
  for (int b = 0; b < nseq; ++b) states[b]->host_pending = n_host[b];
  return EVS_OK;
}

extern "C" int evs_verify_block_trace(evs_state* s, const int32_t* tokens, int32_t n, float* logits,
                                      float* x_trace, cudaStream_t stream) {
  if (!s || !tokens || !logits || !x_trace) return fail(EVS_ERR_ARG, "null argument");
  EVS_TRY(check_block(s, n));
  LaunchCtx Lc{stream, false};
  EVS_TRY(enqueue_verify(s, tokens, n, logits, Lc, x_trace));
  s->host_pending = n;
  return EVS_OK;
}

extern "C" int evs_probs(const float* logits, int32_t n, int32_t V, float T, int32_t top_k, float* p,
                         cudaStream_t stream) {
  if (!logits || !p) return fail(EVS_ERR_ARG, "null argument");
  if (n < 1 || n > 4096 || V < 1 || V > 8192) return fail(EVS_ERR_ARG, "n or V out of range");
  if (!(T > 0.f)) return fail(EVS_ERR_ARG, "temperature must be > 0");
  LaunchCtx Lc{stream, false};
  CUDA_TRY(launch_probs(Lc, logits, n, V, T, top_k, p));
  return EVS_OK;
}

extern "C" int evs_accept(const float* p, const float* q, const int32_t* drafts, const float* u, int32_t n,
                          int32_t V, int32_t mode, int32_t* acc, int32_t* tok, cudaStream_t stream) {
  if (!p || !acc || !tok) return fail(EVS_ERR_ARG, "null argument");
  if (n < 1 || V < 1 || V > 8192) return fail(EVS_ERR_ARG, "n or V out of range");
  if (mode != EVS_GREEDY && mode != EVS_SAMPLE) return fail(EVS_ERR_ARG, "mode must be EVS_GREEDY or EVS_SAMPLE");
  if (n > 1 && !drafts) return fail(EVS_ERR_ARG, "null drafts");
  if (mode == EVS_SAMPLE && (!u || (n > 1 && !q))) return fail(EVS_ERR_ARG, "sample mode needs q and u");
  LaunchCtx Lc{stream, false};
  CUDA_TRY(launch_accept(Lc, p, q, drafts, u, n, V, mode, acc, tok));
  return EVS_OK;
}

extern "C" int evs_markov_draft(const float* trunk, const float* markov, int32_t V, const int32_t* prev,
                                const float* u, int32_t gamma, float T, int32_t top_k, int32_t mode, int32_t* drafts,
                                float* q, cudaStream_t stream) {
  if (!trunk || !markov || !prev || !drafts || !q) return fail(EVS_ERR_ARG, "null argument");
  if (V < 1 || V > 8192 || gamma < 1 || gamma > 64) return fail(EVS_ERR_ARG, "V or gamma out of range");
  if (mode != EVS_GREEDY && mode != EVS_SAMPLE) return fail(EVS_ERR_ARG, "mode must be EVS_GREEDY or EVS_SAMPLE");
  if (mode == EVS_SAMPLE && !u) return fail(EVS_ERR_ARG, "sample mode needs u");
  if (!(T > 0.f)) return fail(EVS_ERR_ARG, "temperature must be > 0");
  LaunchCtx Lc{stream, false};
  CUDA_TRY(launch_markov_draft(Lc, trunk, markov, V, prev, u, gamma, T, top_k, mode, drafts, q));
  return EVS_OK;
}

extern "C" int evs_commit(evs_state* s, int32_t keep, cudaStream_t stream) {
  if (!s) return fail(EVS_ERR_ARG, "null state");
  if (!s->host_pending) return fail(EVS_ERR_STATE, "commit without a pending verify");
  if (keep < 0 || keep > s->host_pending) return fail(EVS_ERR_ARG, "keep=%d outside [0, %d]", keep, s->host_pending);
  LaunchCtx Lc{stream, false};
  CUDA_TRY(launch_commit(Lc, s->book, keep, nullptr, 0));
  s->host_pos += keep;
  s->host_pending = 0;
  return EVS_OK;
}

extern "C" int evs_commit_dev(evs_state* s, const int32_t* accepted, cudaStream_t stream) {
  if (!s || !accepted) return fail(EVS_ERR_ARG, "null argument");
  if (!s->host_pending) return fail(EVS_ERR_STATE, "commit without a pending verify");
  LaunchCtx Lc{stream, false};
  CUDA_TRY(launch_commit(Lc, s->book, 0, accepted, 0));
  s->host_pos_known = false;
  s->host_pending = 0;
  return EVS_OK;
}

extern "C" int evs_round(evs_state* s, const int32_t* tokens, int32_t n, float* logits, float* p, const float* q,
                         const float* u, float T, int32_t top_k, int32_t mode, int32_t* acc, int32_t* otok,
                         cudaStream_t stream) {
  if (!s || !tokens || !logits || !acc || !otok) return fail(EVS_ERR_ARG, "null argument");
  if (mode != EVS_GREEDY && mode != EVS_SAMPLE) return fail(EVS_ERR_ARG, "bad mode");
  if (mode == EVS_SAMPLE && (!p || !u || (n > 1 && !q) || !(T > 0.f)))
    return fail(EVS_ERR_ARG, "sample mode needs p, q, u and T > 0");
  EVS_TRY(check_block(s, n));
  RoundArgs r{p, q, tokens + 1, u, T, top_k, mode, acc, otok};
  GraphEntry key{};
  key.round = true;
  key.n = n;
  key.tok = tokens;
  key.logits = logits;
  key.p = p;
  key.q = q;
  key.u = u;
  key.T = T;
  key.top_k = top_k;
  key.mode = mode;
  key.acc = acc;
  key.otok = otok;
  EVS_TRY(run_captured(s, key, stream, [&](const LaunchCtx& Lc) { return enqueue_round(s, tokens, n, logits, r, Lc); }));
  s->host_pos_known = false;
  s->host_pending = 0;
  return EVS_OK;
}

extern "C" int evs_round_host(evs_state* s, const int32_t* tokens_host, int32_t n, float* logits, float* p,
                              const float* q, const float* u, float T, int32_t top_k, int32_t mode,
                              int32_t* accepted_host, int32_t* token_host, cudaStream_t stream) {
  if (!s || !tokens_host || !logits || !accepted_host || !token_host) return fail(EVS_ERR_ARG, "null argument");
  if (mode != EVS_GREEDY && mode != EVS_SAMPLE) return fail(EVS_ERR_ARG, "bad mode");
  if (mode == EVS_SAMPLE && (!p || !u || (n > 1 && !q) || !(T > 0.f)))
    return fail(EVS_ERR_ARG, "sample mode needs p, q, u and T > 0");
  if (n < 1 || n > NTOK) return fail(EVS_ERR_ARG, "n must be in [1, %d]", NTOK);
  EVS_TRY(check_block(s, n));
  // the staging is free: every call returns after its graph has finished
  memcpy(s->io_pinned, tokens_host, sizeof(int32_t) * n);
  int32_t* tok_d = s->io_dev;
  int32_t* res_d = s->io_dev + NTOK;  // accepted, token
  RoundArgs r{p, q, tok_d + 1, u, T, top_k, mode, res_d, res_d + 1};
  GraphEntry key{};
  key.round = true;
  key.host_io = true;
  key.n = n;
  key.tok = tok_d;
  key.logits = logits;
  key.p = p;
  key.q = q;
  key.u = u;
  key.T = T;
  key.top_k = top_k;
  key.mode = mode;
  key.acc = res_d;
  key.otok = res_d + 1;
  const int rc = run_captured(s, key, stream, [&](const LaunchCtx& Lc) -> int {
    CUDA_TRY(cudaMemcpyAsync(tok_d, s->io_pinned, sizeof(int32_t) * n, cudaMemcpyHostToDevice, Lc.stream));
    EVS_TRY(enqueue_round(s, tok_d, n, logits, r, Lc));
    CUDA_TRY(cudaMemcpyAsync(s->io_pinned + NTOK, res_d, 2 * sizeof(int32_t), cudaMemcpyDeviceToHost, Lc.stream));
    return EVS_OK;
  });
  if (rc != EVS_OK) {
    // without graphs the token copy may already be queued when a later step
    // fails: wait for it, so the next call may rewrite the staging
    cudaStreamSynchronize(stream);
    return rc;
  }
  s->host_pos_known = false;
  s->host_pending = 0;
  CUDA_TRY(cudaStreamSynchronize(stream));
  accepted_host[0] = s->io_pinned[NTOK];
  token_host[0] = s->io_pinned[NTOK + 1];
  return EVS_OK;
}

extern "C" int evs_round_batch(evs_state* const* states, int32_t nseq, const int32_t* tokens, const int32_t* n_host,
                               float* logits, float* p, const float* q, const float* u, float T, int32_t top_k,
                               int32_t mode, int32_t* acc, int32_t* otok, cudaStream_t stream) {
  if (!states || !tokens || !n_host || !logits || !acc || !otok) return fail(EVS_ERR_ARG, "null argument");
  if (mode != EVS_GREEDY && mode != EVS_SAMPLE) return fail(EVS_ERR_ARG, "bad mode");
  if (mode == EVS_SAMPLE && (!p || !u || !q || !(T > 0.f))) return fail(EVS_ERR_ARG, "sample mode needs p, q, u and T > 0");
  SeqRows sr{};
  EVS_TRY(check_batch(states, nseq, n_host, &sr));
  const evs_model* m = states[0]->m;
  const int V = m->cfg.vocab;
  if (V > 8192) return fail(EVS_ERR_UNSUPPORTED, "accept needs V <= 8192");
  RoundArgs r{p, q, tokens + 1, u, T, top_k, mode, acc, otok};
  GraphEntry key{};
  key.round = true;
  key.n = sr.row0[nseq];
  key.tok = tokens;
  key.logits = logits;
  key.p = p;
  key.q = q;
  key.u = u;
  key.T = T;
  key.top_k = top_k;
  key.mode = mode;
  key.acc = acc;
  key.otok = otok;
  key.nseq = nseq;
  for (int b = 0; b < nseq; ++b) {
    key.uid[b] = states[b]->uid;
    key.ns[b] = n_host[b];
  }
  EVS_TRY(run_captured(states[0], key, stream,
                       [&](const LaunchCtx& Lc) { return enqueue_round_batch(states, sr, tokens, logits, r, Lc); }));
  for (int b = 0; b < nseq; ++b) {
    states[b]->host_pos_known = false;
    states[b]->host_pending = 0;
  }
  return EVS_OK;
}

// =================================================================== operators
extern "C" int evs_op_fir(int32_t L, int32_t d, int32_t n, int32_t n_max, int32_t dtype, const void* abv,
                          const float* taps, float* ring, const evs_book* book, void* g, cudaStream_t stream) {
  if (!abv || !taps || !ring || !book || !g) return fail(EVS_ERR_ARG, "null argument");
  if (L < 1 || L > 256 || d < 32 || d % 32 || n < 1 || n > NTOK || n > n_max)
    return fail(EVS_ERR_ARG, "bad FIR shape");
  if (dtype != EVS_BF16 && dtype != EVS_F32) return fail(EVS_ERR_ARG, "bad dtype");
  LaunchCtx Lc{stream, false};
  CUDA_TRY(launch_fir(Lc, dtype, MixSrc{abv, 3 * d, dtype == EVS_F32}, d, one_seq(n), L, L - 1 + n_max, taps,
                      one_ptr(ring), one_ptr(book), g));
  return EVS_OK;
}

extern "C" int evs_op_iir(int32_t M, int32_t d, int32_t n, int32_t n_max, int32_t dtype, const void* abv,
                          const float* lam, const float* res, float* s0, float* s1, const evs_book* book, void* g,
                          cudaStream_t stream) {
  if (!abv || !lam || !res || !s0 || !s1 || !book || !g) return fail(EVS_ERR_ARG, "null argument");
  if (M < 1 || M > 32 || (M & (M - 1)) || d % (256 / M) || n < 1 || n > NTOK || n > n_max)
    return fail(EVS_ERR_ARG, "bad IIR shape");
  if (dtype != EVS_BF16 && dtype != EVS_F32) return fail(EVS_ERR_ARG, "bad dtype");
  LaunchCtx Lc{stream, false};
  CUDA_TRY(launch_iir(Lc, dtype, MixSrc{abv, 3 * d, dtype == EVS_F32}, d, one_seq(n), M, lam, res, one_ptr(s0),
                      one_ptr(s1), one_ptr(book), g));
  return EVS_OK;
}

extern "C" size_t evs_op_attention_scratch_bytes(int32_t H, int32_t Dh, int64_t ctx_max, int32_t chunk, int32_t n_max) {
  (void)n_max;
  if (H < 1 || Dh < 2 || ctx_max < 1 || chunk < 1) return 0;
  return attn_scratch_bytes(H, Dh, ctx_max, chunk);
}

extern "C" int evs_op_attention(int32_t H, int32_t Dh, int32_t n, int32_t n_max, int64_t ctx_max, int32_t chunk,
                                float base, int32_t dtype, const void* qkv, void* kc, void* vc, evs_book* book,
                                void* g, void* scratch, size_t scratch_bytes, cudaStream_t stream) {
  if (!qkv || !kc || !vc || !book || !g || !scratch) return fail(EVS_ERR_ARG, "null argument");
  if (H < 1 || (Dh != 32 && Dh != 64 && Dh != 128) || n < 1 || n > NTOK || n > n_max || ctx_max < 1 ||
      (chunk != 32 && chunk != 64 && chunk != 128 && chunk != 256))
    return fail(EVS_ERR_ARG, "bad attention shape");
  if (dtype != EVS_BF16 && dtype != EVS_F32) return fail(EVS_ERR_ARG, "bad dtype");
  if (scratch_bytes < attn_scratch_bytes(H, Dh, ctx_max, chunk)) return fail(EVS_ERR_ARG, "scratch too small");
  int sms = 0;
  EVS_TRY(num_sms_current(&sms));
  AttnBufs B;
  attn_bufs_from_scratch(scratch, H, Dh, ctx_max, chunk, &B);
  LaunchCtx Lc{stream, false};
  CUDA_TRY(fill_rope_table(B, Dh, base, stream));
  AttnSeq as{};
  as.kc.p[0] = kc;
  as.vc.p[0] = vc;
  if (attn_tma_eligible(dtype, H, Dh, ctx_max)) {
    // tensor maps of the caller's caches into the scratch (synchronous: the
    // host copies live on this stack frame)
    CUtensorMap maps[2];
    char err[256] = {0};
    if (!encode_kv_maps(&maps[0], &maps[1], kc, vc, H, Dh, ctx_max, err, sizeof err))
      return fail(EVS_ERR_ARG, "KV tensor map: %s", err);
    CUDA_TRY(cudaMemcpyAsync(B.maps, maps, sizeof maps, cudaMemcpyHostToDevice, stream));
    CUDA_TRY(cudaMemsetAsync(B.arrivals, 0, sizeof(int) * H, stream));
    CUDA_TRY(cudaStreamSynchronize(stream));
    as.kmap.p[0] = B.maps;
    as.vmap.p[0] = B.maps + 1;
    as.arrivals.p[0] = B.arrivals;
  }
  as.book.p[0] = book;
  as.part_o.p[0] = B.part_o;
  as.part_ml.p[0] = B.part_ml;
  (void)sms;
  CUDA_TRY(launch_attention(Lc, dtype, MixSrc{qkv, 3 * H * Dh, dtype == EVS_F32}, H, Dh, one_seq(n), ctx_max, chunk,
                            as, B, g));
  return EVS_OK;
}

extern "C" int evs_op_commit(evs_book* book, int32_t keep, int32_t n, cudaStream_t stream) {
  if (!book) return fail(EVS_ERR_ARG, "null book");
  if (n < 1 || keep < 0 || keep > n) return fail(EVS_ERR_ARG, "keep=%d outside [0, n=%d]", keep, n);
  LaunchCtx Lc{stream, false};
  CUDA_TRY(launch_commit(Lc, book, keep, nullptr, n));
  return EVS_OK;
}

// Operator GEMM scratch: [partial slots][slot table][arrival counters][error flag],
// each part 256-byte aligned.  The stream-K plan is sized; the tensor-core
// path may use the (slot-free) cluster plan within the same scratch.
static int gemm_plan_op(int32_t N, int32_t K, bool cluster_ok, GemmPlan* g, size_t* table_off, size_t* total) {
  int sms = 0;
  EVS_TRY(num_sms_current(&sms));
  if (!plan_gemm(N, K, sms, g)) return fail(EVS_ERR_UNSUPPORTED, "GEMM shape %d x %d unsupported", N, K);
  auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
  *table_off = al(partials_bytes(*g));
  *total = *table_off + 2 * al(table_bytes(*g)) + 256;
  const int cl = cluster_ok ? gemm_cluster_choice(N, K, sms) : 0;
  if (cl && !plan_gemm_cluster(N, K, cl, g)) return fail(EVS_ERR_UNSUPPORTED, "GEMM shape %d x %d unsupported", N, K);
  return EVS_OK;
}

extern "C" size_t evs_op_gemm_scratch_bytes(int32_t N, int32_t K, int32_t dtype) {
  (void)dtype;
  if (N < 1 || K < 1) return 0;
  static thread_local GemmPlan g;
  size_t toff = 0, total = 0;
  if (gemm_plan_op(N, K, false, &g, &toff, &total) != EVS_OK) return 0;
  return total;
}

extern "C" int evs_op_gemm(const void* W, const void* X, int32_t N, int32_t K, int32_t n, int32_t dtype, float* Y,
                           void* scratch, size_t scratch_bytes, cudaStream_t stream) {
  if (!W || !X || !Y || !scratch) return fail(EVS_ERR_ARG, "null argument");
  if (N < 1 || K < 1 || n < 1 || n > NTOK) return fail(EVS_ERR_ARG, "bad GEMM shape");
  if (dtype != EVS_BF16 && dtype != EVS_F32) return fail(EVS_ERR_ARG, "bad dtype");
  static thread_local GemmPlan g;
  size_t toff = 0, total = 0;
  const bool tc = dtype == EVS_BF16 && N % TILE_M == 0 && K % TILE_K == 0 && aligned16(W) && aligned16(X);
  EVS_TRY(gemm_plan_op(N, K, tc, &g, &toff, &total));
  if (scratch_bytes < total) return fail(EVS_ERR_ARG, "scratch too small (%zu < %zu)", scratch_bytes, total);
  Partials P = g.P;
  P.ws = (float*)scratch;
  P.tab = (const int4*)((char*)scratch + toff);
  const size_t tb = (table_bytes(g) + 255) & ~(size_t)255;
  P.cnt = (int*)((char*)scratch + toff + tb);
  P.mode = GEMM_FINAL;
  P.n = n;
  P.fin = Y;
  P.fin_ld = N;
  int* err_flag = (int*)((char*)scratch + total - 256);
  CUDA_TRY(cudaMemcpyAsync((void*)P.tab, g.tab, table_bytes(g), cudaMemcpyHostToDevice, stream));
  CUDA_TRY(cudaMemsetAsync(P.cnt, 0, tb, stream));
  CUDA_TRY(cudaStreamSynchronize(stream));  // g is reused by the next call
  LaunchCtx Lc{stream, false};
  if (tc) {
    CUtensorMap wm, xm;
    char err[256] = {0};
    if (!encode_tmap_2d(&wm, W, K, N, TILE_K, TILE_M, err, sizeof err) ||
        !encode_tmap_2d(&xm, X, K, n, TILE_K, NTOK, err, sizeof err))
      return fail(EVS_ERR_CUDA, "%s", err);
    CUDA_TRY(cudaMemsetAsync(err_flag, 0, sizeof(int), stream));
    CUDA_TRY(launch_gemm_tc(Lc, wm, xm, wm, P, K, err_flag));  // P.pf_units = 0: no prefetch
  } else {
    CUDA_TRY(launch_gemm_simt(Lc, dtype, W, X, K, P, K));
  }
  return EVS_OK;
}

// ------------------------------------------- operator GEMM, static scratch
// evs_op_gemm for callers that must not allocate device memory on their
// path: a serving loop that forbids allocation once it runs (an allocation
// can synchronize the device and fail when memory is fragmented), or a
// plug-in whose host framework owns all device memory and hands it no
// scratch.  Its scratch ([partial slots][slot table][arrival counters][error
// flag], as evs_op_gemm lays it out) is this file-scope device array, one per
// device; calls that overlap in time share it and race.
constexpr size_t STATIC_GEMM_SCRATCH = EVS_OP_GEMM_STATIC_SCRATCH_BYTES;
static __device__ __align__(256) uint8_t g_static_gemm_scratch[STATIC_GEMM_SCRATCH];

// The array's device address, looked up once per device.  The first lookup
// may load the module, so the first call on a device belongs outside
// stream capture.
static int static_gemm_scratch(void** out) {
  static std::mutex mu;
  static void* addr[64] = {};
  int dev = 0;
  CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return fail(EVS_ERR_UNSUPPORTED, "device ordinal %d", dev);
  std::lock_guard<std::mutex> lk(mu);
  if (!addr[dev]) CUDA_TRY(cudaGetSymbolAddress(&addr[dev], g_static_gemm_scratch));
  *out = addr[dev];
  return EVS_OK;
}

extern "C" int evs_op_gemm_static(const void* W, const void* X, int32_t N, int32_t K, int32_t n, int32_t dtype,
                                  float* Y, cudaStream_t stream) {
  if (!W || !X || !Y) return fail(EVS_ERR_ARG, "null argument");
  if (N < 1 || K < 1 || n < 1 || n > NTOK) return fail(EVS_ERR_ARG, "bad GEMM shape");
  if (dtype != EVS_BF16 && dtype != EVS_F32) return fail(EVS_ERR_ARG, "bad dtype");
  static thread_local GemmPlan g;
  size_t toff = 0, total = 0;
  const bool tc = dtype == EVS_BF16 && N % TILE_M == 0 && K % TILE_K == 0 && aligned16(W) && aligned16(X);
  EVS_TRY(gemm_plan_op(N, K, tc, &g, &toff, &total));
  if (total > STATIC_GEMM_SCRATCH)
    return fail(EVS_ERR_CAPACITY, "GEMM %d x %d needs %zu bytes of scratch; the static array holds %zu", N, K, total,
                STATIC_GEMM_SCRATCH);
  void* scratch = nullptr;
  EVS_TRY(static_gemm_scratch(&scratch));
  Partials P = g.P;
  P.ws = (float*)scratch;
  P.tab = (const int4*)((char*)scratch + toff);
  const size_t tb = (table_bytes(g) + 255) & ~(size_t)255;
  P.cnt = (int*)((char*)scratch + toff + tb);
  P.mode = GEMM_FINAL;
  P.n = n;
  P.fin = Y;
  P.fin_ld = N;
  int* err_flag = (int*)((char*)scratch + total - 256);
  // arrival counters and error flag start at zero (memsets, no allocation);
  // the partial slots need no initial value
  CUDA_TRY(cudaMemcpyAsync((void*)P.tab, g.tab, table_bytes(g), cudaMemcpyHostToDevice, stream));
  CUDA_TRY(cudaMemsetAsync(P.cnt, 0, tb, stream));
  CUDA_TRY(cudaMemsetAsync(err_flag, 0, sizeof(int), stream));
  CUDA_TRY(cudaStreamSynchronize(stream));  // g is reused by the next call
  LaunchCtx Lc{stream, false};
  if (tc) {
    CUtensorMap wm, xm;
    char err[256] = {0};
    if (!encode_tmap_2d(&wm, W, K, N, TILE_K, TILE_M, err, sizeof err) ||
        !encode_tmap_2d(&xm, X, K, n, TILE_K, NTOK, err, sizeof err))
      return fail(EVS_ERR_CUDA, "%s", err);
    CUDA_TRY(launch_gemm_tc(Lc, wm, xm, wm, P, K, err_flag));
  } else {
    CUDA_TRY(launch_gemm_simt(Lc, dtype, W, X, K, P, K));
  }
  // The flag lives in the library's array, out of the caller's reach: read
  // it back here (a 4-byte copy into this stack frame, no allocation) so a
  // pipeline wait that gave up is reported by this call.
  int flag = 0;
  CUDA_TRY(cudaMemcpyAsync(&flag, err_flag, sizeof(int), cudaMemcpyDeviceToHost, stream));
  CUDA_TRY(cudaStreamSynchronize(stream));
  if (flag) return fail(EVS_ERR_DEVICE, "device status 0x%x (a GEMM pipeline wait gave up; Y is incomplete)", flag);
  return EVS_OK;
}

// =================================================================== profiling
namespace {

// One weight GEMM of a verify step as the step launches it (B source and
// output mode), for the profiling entry points.
struct GemmCall {
  const Partials* plan;
  const CUtensorMap *wm, *xm;
  const uint8_t* pk;
  const void *W, *X;
  int N, K, bsrc, mode;
};

// The step's GEMMs in order: per layer in, out, gate/up, down; then the head.
// Outputs go to scratch and residual GEMMs write plain sums (or slots), so
// the decoding state is untouched.
std::vector<GemmCall> step_gemms(evs_state* s) {
  const evs_model* m = s->m;
  const evs_config& c = m->cfg;
  const int d = c.d_model, F = c.d_ffn, V = c.vocab;
  const bool fz = m->fuse;
  auto slots_or = [&](const Partials& P, bool resid, int mode) {
    return m->slots && P.cl == 0 && P.max_cnt <= (resid ? SLOTS_RESID_MAX : SLOTS_MIX_MAX) &&
                   !(resid && (fz || !m->slots_resid))
               ? GEMM_SLOTS
               : mode;
  };
  std::vector<GemmCall> v;
  for (size_t i = 0; i < m->L.size(); ++i) {
    const LayerW& w = m->L[i];
    const bool nin = fz && i > 0;
    v.push_back({&m->p_in, &w.m_in, nin ? &s->m_xf : &s->m_xn, w.pk_in, w.w_in, nin ? (const void*)s->X : s->xn,
                 3 * d, d, nin ? GEMM_B_NORM : GEMM_B_TMA, slots_or(m->p_in, false, GEMM_FINAL)});
    v.push_back({&m->p_out, &w.m_out, &s->m_g, w.pk_out, w.w_out, s->g, d, d, GEMM_B_TMA,
                 slots_or(m->p_out, true, GEMM_FINAL)});
    v.push_back({&m->p_gu, &w.m_gu, fz ? &s->m_xf : &s->m_xn, w.pk_gu, w.w_gu, fz ? (const void*)s->X : s->xn,
                 2 * F, d, fz ? GEMM_B_NORM : GEMM_B_TMA,
                 m->swiglu ? GEMM_SWIGLU : slots_or(m->p_gu, false, GEMM_FINAL)});
    v.push_back({&m->p_down, &w.m_down, &s->m_h, w.pk_down, w.w_down, s->h, d, F, GEMM_B_TMA,
                 slots_or(m->p_down, true, GEMM_FINAL)});
  }
  v.push_back({&m->p_head, &m->m_head, fz ? &s->m_xf : &s->m_xn, m->pk_head, m->head,
               fz ? (const void*)s->X : s->xn, V, d, fz ? GEMM_B_NORM : GEMM_B_TMA, GEMM_FINAL});
  return v;
}

// Launches call k of calls; with chain, it warms L2 with the first units of
// call k + 1 (the next weight matrix) as the verify step does.
int launch_profiled(evs_state* s, const std::vector<GemmCall>& calls, size_t k, int n, bool chain,
                    const LaunchCtx& Lc, int64_t* bytes) {
  const evs_model* m = s->m;
  const evs_config& c = m->cfg;
  const GemmCall& g = calls[k];
  const size_t es = esize(c.dtype);
  Partials P = *g.plan;
  P.nt = 1;
  P.wpk = g.pk;
  P.bsrc = g.bsrc;
  P.Kdim = g.K;
  P.ss_in = s->ss;
  P.ss_tiles = (c.d_model + TILE_M - 1) / TILE_M;
  P.norm_d = c.d_model;
  P.eps = c.norm_eps;
  P.hout = reinterpret_cast<bf16*>(s->pout);
  P.h_cols = c.d_ffn;
  P.ws = s->ws[k & 1];
  P.cnt = s->cnt;
  P.mode = g.mode;
  P.n = n;
  P.fin = s->pout;
  P.fin_ld = g.N;
  const CUtensorMap* nmap = g.wm;
  if (chain) {
    const GemmCall& nx = calls[(k + 1) % calls.size()];
    nmap = nx.wm;
    P.nwpk = nx.pk;
    P.pf_units = s->pf_units;
    P.nG = nx.plan->G;
    P.nKB = nx.plan->KB;
    P.nU = nx.plan->U;
    P.ncl = nx.plan->cl;
  }
  if (m->tc)
    CUDA_TRY(launch_gemm_tc(Lc, *g.wm, *g.xm, *nmap, P, g.K, &s->book->status));
  else
    CUDA_TRY(launch_gemm_simt(Lc, c.dtype, g.W, g.X, g.K, P, g.K));
  const int64_t in_es = g.bsrc == GEMM_B_TMA ? (int64_t)es : 4;
  const int64_t out_b = g.mode == GEMM_SWIGLU ? (int64_t)n * (g.N / 2) * 2 : (int64_t)n * g.N * 4;
  *bytes = (int64_t)g.N * g.K * es + (int64_t)n * g.K * in_es + out_b;
  return EVS_OK;
}

}  // namespace

extern "C" int evs_profile_gemms(evs_state* s, int32_t n, float* ms_host, int64_t* bytes_host, int32_t max_launches,
                                 int32_t* count, cudaStream_t stream) {
  if (!s || !ms_host || !bytes_host || !count) return fail(EVS_ERR_ARG, "null argument");
  if (n < 1 || n > s->m->n_max) return fail(EVS_ERR_ARG, "n out of range");
  const std::vector<GemmCall> calls = step_gemms(s);
  const int total = (int)calls.size();
  if (max_launches < total) return fail(EVS_ERR_ARG, "need room for %d launches", total);
  std::vector<cudaEvent_t> ev(total + 1);
  for (auto& e : ev) CUDA_TRY(cudaEventCreate(&e));
  LaunchCtx Lc{stream, false};
  // keep the GPU busy while the host enqueues, so events time only the GEMMs
  CUDA_TRY(launch_busy(Lc, 2000000));
  int r = EVS_OK;
  int k = 0;
  for (; k < total && r == EVS_OK; ++k) {
    cudaError_t e = cudaEventRecord(ev[k], stream);
    if (e != cudaSuccess) r = fail(EVS_ERR_CUDA, "profiling events: %s", cudaGetErrorString(e));
    if (r == EVS_OK) r = launch_profiled(s, calls, k, n, false, Lc, &bytes_host[k]);
  }
  if (r == EVS_OK) {
    cudaError_t e = cudaEventRecord(ev[k], stream);
    if (e == cudaSuccess) e = cudaEventSynchronize(ev[k]);
    for (int j = 0; j < k && e == cudaSuccess; ++j) e = cudaEventElapsedTime(&ms_host[j], ev[j], ev[j + 1]);
    if (e != cudaSuccess) r = fail(EVS_ERR_CUDA, "profiling events: %s", cudaGetErrorString(e));
  }
  for (auto& e : ev) cudaEventDestroy(e);
  *count = k;
  return r;
}

extern "C" int evs_profile_gemm_chain(evs_state* s, int32_t n, int32_t reps, float* ms_per_chain,
                                      int64_t* bytes_per_chain, int32_t* launches, cudaStream_t stream) {
  if (!s || !ms_per_chain || !bytes_per_chain || !launches) return fail(EVS_ERR_ARG, "null argument");
  if (n < 1 || n > s->m->n_max || reps < 1 || reps > 1000) return fail(EVS_ERR_ARG, "n or reps out of range");
  const std::vector<GemmCall> calls = step_gemms(s);
  // the chain as one graph with programmatic dependent launch between GEMMs
  int64_t bytes = 0;
  const long long before = g_launches.load();
  CUDA_TRY(cudaStreamBeginCapture(s->cap, cudaStreamCaptureModeRelaxed));
  LaunchCtx Lc{s->cap, s->pdl};
  int r = EVS_OK;
  for (size_t k = 0; k < calls.size() && r == EVS_OK; ++k) {
    int64_t b = 0;
    r = launch_profiled(s, calls, k, n, true, Lc, &b);
    bytes += b;
  }
  cudaGraph_t graph = nullptr;
  cudaError_t e = cudaStreamEndCapture(s->cap, &graph);
  g_launches -= g_launches.load() - before;  // captured, not launched: counted per graph launch below
  if (r != EVS_OK) {
    if (graph) cudaGraphDestroy(graph);
    return r;
  }
  if (e != cudaSuccess) return fail(EVS_ERR_CUDA, "stream capture failed: %s", cudaGetErrorString(e));
  cudaGraphExec_t exec = nullptr;
  e = cudaGraphInstantiate(&exec, graph, 0);
  cudaGraphDestroy(graph);
  if (e != cudaSuccess) return fail(EVS_ERR_CUDA, "graph instantiate failed: %s", cudaGetErrorString(e));
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  e = cudaEventCreate(&e0);
  if (e == cudaSuccess) e = cudaEventCreate(&e1);
  for (int i = 0; i < 3 && e == cudaSuccess; ++i) e = cudaGraphLaunch(exec, stream);  // warm-up
  if (e == cudaSuccess) e = cudaEventRecord(e0, stream);
  for (int i = 0; i < reps && e == cudaSuccess; ++i) e = cudaGraphLaunch(exec, stream);
  if (e == cudaSuccess) e = cudaEventRecord(e1, stream);
  if (e == cudaSuccess) e = cudaEventSynchronize(e1);
  float ms = 0.f;
  if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  cudaGraphExecDestroy(exec);
  if (e != cudaSuccess) return fail(EVS_ERR_CUDA, "chain timing: %s", cudaGetErrorString(e));
  count_launch((long long)(reps + 3) * (long long)calls.size());
  *ms_per_chain = ms / reps;
  *bytes_per_chain = bytes;
  *launches = (int32_t)calls.size();
  return EVS_OK;
}

extern "C" int evs_selftest_wait_timeout(int32_t* status_dev, int64_t limit_ns, cudaStream_t stream) {
  if (!status_dev) return fail(EVS_ERR_ARG, "null status");
  if (limit_ns < 1000 || limit_ns > 1000000000) return fail(EVS_ERR_ARG, "limit_ns outside [1e3, 1e9]");
  CUDA_TRY(launch_wait_selftest(stream, status_dev, (unsigned long long)limit_ns));
  return EVS_OK;
}

// =================================================================== misc
extern "C" const char* evs_last_error(void) { return g_err.c_str(); }
extern "C" const char* evs_version(void) { return "evs 0.1 (sm_103a)"; }
extern "C" int64_t evs_kernel_launches(void) { return g_launches.load(); }
extern "C" int32_t evs_verify_kernel_count(const evs_state* s, int32_t n) {
  (void)n;
  if (!s) return -1;
  const evs_config& c = s->m->cfg;
  const int ak = attn_kernels(c.dtype, c.n_heads, c.head_dim, s->ctx_max);
  if (s->use_engine) {
    // embed, one engine launch per span, the attention kernels of each attention layer
    int k = 1 + (int)s->eng_segs.size();
    for (const auto& L : s->m->L) k += L.kind == EVS_LAYER_ATTN ? ak : 0;
    return k;
  }
  int k = 1 + 2;  // embed, head GEMM, logits
  // per layer: 4 GEMMs + the mixer (2 or 3 kernels for attention), plus two
  // RMSNorm kernels and the activation kernel unless the GEMMs do that work
  for (const auto& L : s->m->L)
    k += 4 + (s->m->fuse ? 0 : 2) + (s->m->swiglu ? 0 : 1) + (L.kind == EVS_LAYER_ATTN ? ak : 1);
  return k;
}
