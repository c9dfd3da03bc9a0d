/*
 * evs.h - C ABI of the block-verify / accept / commit path of lossless
 * speculative decoding for StripedHyena2-style hybrid models (EvSpark).
 *
 * Sources (cited by page and passage):
 *  [abstract]    "EvSpark: Lossless Speculative Decoding for Hybrid DNA
 *                Foundation Models", preprint abstract, contribution (i):
 *                block-verification forward pass + per-position state-slicing
 *                rollback over FIR windows, IIR recurrences and KV caches,
 *                with zero recomputation; exact rejection-sampling verify.
 *  [systems]     GitHub discussion "EvSpark: ~3x lossless speculative decoding
 *                for Evo2 7B with hybrid-state rollback", "The systems
 *                problem": KV caches append-only, FIR states fixed-length
 *                sliding windows, IIR states recurrent over the whole prefix.
 *  [implemented] same post, "What we implemented": keep the intermediate
 *                state of every block position, slice to the accepted
 *                boundary once the verifier decides.
 *  [prereq1]     same discussion, author's reply, prerequisite 1: the
 *                per-position FIR/IIR state of all gamma+1 candidates.
 *  [library]     model card "EvSpark - lossless speculative decoding for
 *                Evo2", "Library" / "Quickstart": generate / generate_native,
 *                greedy, T = 1.0, top_k = 4, decode-time gamma' <= gamma.
 *
 * Conventions
 *  - Every function returns EVS_OK (0) or an EVS_ERR_* code; the message of
 *    the last failure on the calling thread is evs_last_error().
 *  - Pointers named *_dev are device pointers (cudaMalloc'd or equivalent,
 *    16-byte aligned); *_host are host pointers.  Inputs and outputs are
 *    owned by the caller; evs_model / evs_state buffers by the library.
 *  - Work is enqueued on the caller's stream and returns without waiting,
 *    unless a function says "synchronous".
 *  - Storage dtype (EVS_BF16 / EVS_F32) applies to weights, GEMM inputs and
 *    the KV cache; residual stream, filter state, logits and probabilities
 *    are always float32.
 *  - In-kernel checks never trap: they set bits of the state's device status
 *    word (EVS_DEV_*), skip the offending access, and evs_state_check()
 *    reports them.
 */
#ifndef EVS_H
#define EVS_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------- codes */
enum {
  EVS_OK = 0,
  EVS_ERR_ARG = 1,         /* bad argument (null, range, alignment, shape) */
  EVS_ERR_STATE = 2,       /* protocol misuse: commit without a pending verify, verify while one is pending */
  EVS_ERR_CAPACITY = 3,    /* committed length + n > ctx_max */
  EVS_ERR_OOM = 4,         /* device allocation failed */
  EVS_ERR_CUDA = 5,        /* a CUDA runtime / driver call failed */
  EVS_ERR_DEVICE = 6,      /* an in-kernel check fired (see EVS_DEV_*) */
  EVS_ERR_UNSUPPORTED = 7  /* shape the kernels do not handle (message says why) */
};

/* bits of evs_book.status */
enum {
  EVS_DEV_BAD_TOKEN = 1,   /* a token id outside [0, vocab) */
  EVS_DEV_KV_OVERFLOW = 2, /* an append past ctx_max */
  EVS_DEV_BAD_KEEP = 4,    /* commit keep outside [0, pending n] */
  EVS_DEV_TIMEOUT = 8,     /* a bounded pipeline wait gave up */
  EVS_DEV_BAD_PROBS = 16   /* a sampled row had no mass (NaN or all entries below 2^-24):
                              its argmax was emitted instead (evs_round / evs_round_batch) */
};

enum { EVS_F32 = 0, EVS_BF16 = 1 };
enum { EVS_LAYER_FIR = 0, EVS_LAYER_IIR = 1, EVS_LAYER_ATTN = 2 };
enum { EVS_GREEDY = 0, EVS_SAMPLE = 1 };

/* ---------------------------------------------------------------- model */
/* Shape of the hybrid stack.  Layer i is
 *   EVS_LAYER_FIR  : Hyena mixer with an explicit causal filter of length
 *                    layer_param[i] in [1, 256] (short / medium FIR, [systems]);
 *   EVS_LAYER_IIR  : Hyena mixer with a modal IIR filter of layer_param[i]
 *                    diagonal complex poles (1..32) ([systems]);
 *   EVS_LAYER_ATTN : multi-head attention with rotary embedding over an
 *                    append-only KV cache; layer_param ignored.
 * Each layer is  x += Mixer(RMSNorm(x)); x += MLP(RMSNorm(x)), with
 * Hyena  [a|b|v] = W_in xn, z = b*v, y = h (*) z, out = W_out (a*y);
 * MLP    W_down (silu(W_gate xn) * W_up xn); head logits = W_lm RMSNorm(x).
 * bf16 storage needs d_model, 2*d_ffn, vocab multiples of 128 and
 * d_model, d_ffn multiples of 64; f32 storage has no such limit.        */
/* Alternative kernel arrangements of the bf16 path, each bit-for-bit equal to
 * the default and measured slower on the 7B-shaped round; for comparison.
 *  EVS_OPT_SWIGLU_EPILOGUE: SiLU-and-multiply in the gate/up GEMM's epilogue
 *    (gate / up rows interleaved by 64 in the packed weights).
 *  EVS_OPT_NORM_IN_GEMM: the RMSNorm of each GEMM input built by the GEMM's
 *    own B-tile converters from the fp32 residual rows (passes of at most
 *    16 rows).
 *  EVS_OPT_GEMM_SUMS_SLOTS: every GEMM sums its split-K partials itself
 *    (the last contributor of a tile; out / down on 4-CTA clusters) instead
 *    of leaving them to the consuming kernel. */
enum { EVS_OPT_SWIGLU_EPILOGUE = 1, EVS_OPT_NORM_IN_GEMM = 2, EVS_OPT_GEMM_SUMS_SLOTS = 4 };

typedef struct evs_config {
  int32_t vocab;
  int32_t d_model;
  int32_t n_layers;
  int32_t n_heads;
  int32_t head_dim;       /* even; n_heads * head_dim == d_model when any attention layer exists */
  int32_t d_ffn;
  int32_t gamma_max;      /* verify blocks hold n <= gamma_max + 1 <= 16 tokens */
  int32_t dtype;          /* EVS_BF16 or EVS_F32 */
  int32_t attn_chunk;     /* keys per split-KV chunk: 32, 64, 128 or 256 */
  float rope_base;        /* e.g. 10000 */
  float norm_eps;         /* e.g. 1e-6 */
  int32_t options;        /* EVS_OPT_* bits, 0 = the default (fastest measured) kernels */
  const int32_t* layer_kind_host;   /* [n_layers] EVS_LAYER_* */
  const int32_t* layer_param_host;  /* [n_layers] */
} evs_config;

/* Device weights, row-major [out][in] in the storage dtype; caller-owned,
 * must stay valid until evs_model_destroy.
 *  w_in   [3*d][d]   rows a|b|v (Hyena) or q|k|v (attention, heads contiguous)
 *  w_out  [d][d]
 *  w_gu   [2*F][d]   rows 0..F-1 gate, F..2F-1 up
 *  w_down [d][F]
 *  fir_taps    float32 [L][d]; tap j multiplies z_{t-j}
 *  iir_lambda  float32 [d][M][2] complex poles (re, im)
 *  iir_residue float32 [d][M][2] complex residues                          */
typedef struct evs_layer_weights {
  const void* w_in;
  const void* w_out;
  const void* w_gu;
  const void* w_down;
  const float* fir_taps;
  const float* iir_lambda;
  const float* iir_residue;
} evs_layer_weights;

typedef struct evs_weights {
  const void* embed;                  /* [vocab][d] */
  const void* lm_head;                /* [vocab][d] */
  const evs_layer_weights* layers_host; /* [n_layers], read during create only */
} evs_weights;

typedef struct evs_model evs_model;
typedef struct evs_state evs_state;

/* Creates a model on the current device.  With bf16 storage it also copies
 * every projection matrix (w_in, w_out, w_gu, w_down, lm_head) into a
 * library-owned device buffer in the GEMM's streaming layout: 16 KB blocks
 * of 128 rows x 64 columns in the order the GEMM reads them, each already in
 * its shared-memory (128-byte swizzled) image, zero-padded at ragged edges.
 * This costs one extra copy of those matrices in device memory and
 * synchronizes the device once.  Returns EVS_ERR_UNSUPPORTED for shapes the
 * kernels lack, EVS_ERR_OOM when the packed copy does not fit. */
int evs_model_create(const evs_config* cfg, const evs_weights* w, evs_model** out);
int evs_model_destroy(evs_model* m);

/* ---------------------------------------------------------------- state */
/* Device-resident bookkeeping of one decoding state.  Commit copies nothing
 * ([implemented]): FIR inputs live in one ring per layer indexed by absolute
 * position, so moving pos moves every window; IIR states live in two banks
 * per layer, a verify reads the current bank and writes its per-position
 * states to the other, and commit flips the bank and picks the slot.     */
typedef struct evs_book {
  int32_t pos;        /* committed tokens = valid KV rows = next position; the
                         FIR input of position p is ring row p mod (L-1+n_max) */
  int32_t reserved0;  /* zero */
  int32_t reserved1;  /* zero */
  int32_t iir_bank;   /* bank holding the current IIR states */
  int32_t iir_slot;   /* slot within that bank, -1 = the zero initial state */
  int32_t pending_n;  /* block size awaiting commit, 0 if none */
  int32_t status;     /* EVS_DEV_* bits */
  int32_t reserved;
} evs_book;

/* Per-layer state buffers (device pointers owned by the state):
 *  FIR : fir_ring  float32 [L-1+n_max][d] - the input z of position p at row
 *        p mod (L-1+n_max); the window of the committed state (the last L-1
 *        inputs) is positions pos-L+1 .. pos-1, zero before position 0.  A
 *        verify of n tokens writes positions pos .. pos+n-1 and leaves the
 *        window of every block position in place.
 *  IIR : iir_all[b]  float32 [n_max][d][M][2] - state after each block position
 *  ATTN: k_cache, v_cache [H][ctx_max][Dh] storage dtype (head-major, so a
 *        head's keys stream contiguously)                               */
typedef struct evs_layer_view {
  int32_t kind, param;
  float* fir_ring;
  void* reserved;
  float* iir_all[2];
  void* k_cache;
  void* v_cache;
  int64_t ctx_max;
  int32_t n_max;
} evs_layer_view;

/* Allocates all state for up to ctx_max positions (KV caches for attention
 * layers, a FIR ring / two IIR banks per Hyena layer, activations,
 * workspaces) and resets it.  Synchronous. */
int evs_state_create(evs_model* m, int64_t ctx_max, evs_state** out);
int evs_state_destroy(evs_state* s);
/* Zero windows / states, empty caches, position 0.  Enqueued on stream. */
int evs_state_reset(evs_state* s, cudaStream_t stream);
/* Copies every buffer and the bookkeeping of src into dst (same model and
 * ctx_max): the snapshot of snapshot-and-replay rollback ([abstract]). */
int evs_state_clone(const evs_state* src, evs_state* dst, cudaStream_t stream);
/* Copies the recurrent state only (FIR windows, IIR modal states) and the
 * bookkeeping of src into dst (same model and ctx_max); the KV caches are
 * not copied: they are append-only, rows below pos never change and rows
 * from pos on are rewritten by the next verify.  This is the snapshot (and,
 * copied back, the restore) of the snapshot-and-replay baseline that
 * per-position state slicing replaces ([abstract], [systems]): snapshot,
 * verify, restore, verify the kept tokens again, commit.  Synchronous read
 * of src's bookkeeping; the copies are enqueued on stream. */
int evs_state_snapshot(const evs_state* src, evs_state* dst, cudaStream_t stream);
int evs_state_layer_view(const evs_state* s, int32_t layer, evs_layer_view* out);
/* Device address of the bookkeeping (for graph-captured callers). */
int evs_state_book_dev(const evs_state* s, evs_book** out);
/* Synchronous read / write of the bookkeeping (tests, synthesised states).
 * A write also updates the host's copy of pos and pending_n. */
int evs_state_book_read(const evs_state* s, evs_book* out_host, cudaStream_t stream);
int evs_state_book_write(evs_state* s, const evs_book* in_host, cudaStream_t stream);
/* Synchronous: waits for the stream, returns EVS_ERR_DEVICE if any
 * EVS_DEV_* bit is set (status copied to *status_host when non-null). */
int evs_state_check(evs_state* s, cudaStream_t stream, int32_t* status_host);
/* Capture verify / commit sequences in CUDA graphs (default on). */
int evs_state_use_graphs(evs_state* s, int32_t enable);
/* Run single-sequence verifies through the persistent engine (off by
 * default; available where the model allows it: bf16 storage, FIR filters of
 * at most 128 taps): one kernel per span of layers between attention
 * mixers, in which the weight GEMMs stream without stopping at layer
 * boundaries and the row work between them (mixers, residual add + RMSNorm,
 * SiLU-and-multiply, logits) runs on other warps of the same CTAs,
 * synchronised through counters in global memory.  Results equal the
 * separate kernels' bit for bit.  On the 7B-shaped stack it is slower than
 * the separate kernels with programmatic dependent launch (3.2 against
 * 2.73 ms per round of 13): each SM takes in weight units at about its
 * share of the HBM bandwidth and no faster, so the stream cannot catch up
 * after a stall, and a layer boundary handed over through global counters
 * takes longer than a kernel boundary.  Traced and batched verifies always
 * use the separate kernels.  EVS_ERR_UNSUPPORTED when enabling it for a
 * model it does not take. */
int evs_state_use_engine(evs_state* s, int32_t enable);

/* ---------------------------------------------------------------- path */
/* Block verify ([abstract] (i); [implemented]; [prereq1]).
 * tokens_dev int32 [n]: the pending token followed by n-1 drafts.
 * Writes logits_dev float32 [n][vocab], row i scoring the token after
 * tokens[i].  Every layer keeps the state after each block position:
 * FIR ext rows, IIR per-position states, KV rows pos..pos+n-1.  n = 1 is
 * native decoding.  1 <= n <= gamma_max+1; EVS_ERR_STATE if a verify is
 * pending; EVS_ERR_CAPACITY if pos + n > ctx_max (pos as known to the host:
 * after evs_commit_dev the device checks and sets EVS_DEV_KV_OVERFLOW). */
int evs_verify_block(evs_state* s, const int32_t* tokens_dev, int32_t n,
                     float* logits_dev, cudaStream_t stream);

/* Batched block verify: one forward pass over the blocks of nseq sequences
 * (the weights are read once for all of them), each sequence keeping its
 * own per-position state for its own later commit (ragged rollback:
 * evs_commit / evs_commit_dev per state) — the batched verify the pages
 * name as the next step for serving ([systems], [regime]).
 * states_host [nseq] (1 <= nseq <= 16): distinct states of one model and one
 * ctx_max, none with a pending verify; n_host [nseq]: block lengths, each in
 * [1, gamma_max+1], summing to at most 128 (EVS_BATCH_ROWS_MAX) on the bf16
 * path, at most 16 for float32 models and with EVS_OPT_NORM_IN_GEMM
 * (EVS_ERR_UNSUPPORTED between 17 and 128); tokens_dev: the blocks back to
 * back (sequence 0's n_host[0] tokens first); logits_dev [sum n][V] in the
 * same row order.  The weight GEMMs take all rows in one pass (16-row
 * chunks side by side in the tensor-core N dimension).  The activations and
 * workspaces of states_host[0] are used.  Each sequence's logits and
 * retained state equal those of its own evs_verify_block bit for bit.
 * Launched directly on stream (not captured in a graph).  Errors as
 * evs_verify_block, per state. */
#define EVS_BATCH_ROWS_MAX 128
int evs_verify_batch(evs_state* const* states_host, int32_t nseq, const int32_t* tokens_dev,
                     const int32_t* n_host, float* logits_dev, cudaStream_t stream);
/* Block verify that also copies the residual stream after the embedding
 * and after every layer to x_trace_dev float32 [n_layers+1][n][d_model]
 * (layer-by-layer validation and tracing; runs without graph capture).
 * Same contract as evs_verify_block otherwise. */
int evs_verify_block_trace(evs_state* s, const int32_t* tokens_dev, int32_t n,
                           float* logits_dev, float* x_trace_dev, cudaStream_t stream);

/* Target distribution ([library]: T, top_k).  logits_dev [n][V] ->
 * p_dev [n][V]: softmax of logits / T over the top_k largest entries of each
 * row (ties to the lower index; a NaN ranks below every number, so it enters
 * the support only when a row holds fewer than top_k numbers), zero
 * elsewhere; top_k <= 0 or >= V keeps all.  T > 0. */
int evs_probs(const float* logits_dev, int32_t n, int32_t V, float T,
              int32_t top_k, float* p_dev, cudaStream_t stream);

/* Accept rule ([abstract]: exact rejection-sampling verification; greedy
 * equality with native decoding).  n = gamma + 1 >= 1 block rows.
 *  p_dev  [n][V]   target rows (greedy: any scores, e.g. logits)
 *  q_dev  [n-1][V] drafter distributions (unused in greedy mode)
 *  drafts_dev int32 [n-1], u_dev float32 [n] uniforms in [0,1) (unused greedy)
 * Draft i (1-based) is accepted iff  greedy: d_i == argmax p_{i-1} (lowest
 * index on ties); sample: u_{i-1} * q_i(d_i) < p_{i-1}(d_i) in float32.
 * At the first rejection a = i-1 and the output token is argmax p_a /
 * sample((p_a - q_{a+1})^+, u_{n-1}) (falls back to p_a if that residual has
 * no integer mass); if all accepted a = n-1 and the token is argmax p_a /
 * sample(p_a, u_{n-1}).  sample(w,u) is the inverse CDF over integer weights
 * floor(w_j 2^24): exact and independent of summation order.  A uniform
 * of 1 or more is taken as the largest float32 below 1.  A row with no
 * integer mass at all (NaN or all entries below 2^-24, never a valid
 * distribution) yields its argmax instead; evs_round / evs_round_batch
 * then also set EVS_DEV_BAD_PROBS in the state's status.
 * Writes out_accepted_dev[0] = a and out_token_dev[0] = token. */
int evs_accept(const float* p_dev, const float* q_dev, const int32_t* drafts_dev,
               const float* u_dev, int32_t n, int32_t V, int32_t mode,
               int32_t* out_accepted_dev, int32_t* out_token_dev, cudaStream_t stream);

/* Drafter-side Markov head ([abstract] (ii): a gamma-parallel drafter trunk
 * with a full-matrix Markov head; model card, drafter description: a full
 * V x V Markov head).  The trunk scores all gamma draft slots in one pass
 * (trunk_logits_dev float32 [gamma][V], e.g. the logits of a verify of the
 * drafter's own stack); the head then draws the drafts one after another:
 * slot i's logits are trunk_logits[i] + markov_dev[prev_i] (row prev_i of
 * float32 [V][V]), prev_0 = prev_dev[0] (the pending token; outside [0, V)
 * selects row 0) and prev_{i+1} = draft i; q_i = softmax over the top_k
 * largest of those logits at temperature T (as evs_probs), written to
 * q_dev [gamma][V]; draft i = sample(q_i, u_dev[i]) with the accept rule's
 * integer-ladder sampler (EVS_SAMPLE; a row without mass gives its argmax)
 * or the argmax of the logits, lowest index on ties (EVS_GREEDY, u_dev
 * unused, may be null), written to drafts_dev[i].  A NaN logit ranks below
 * every number (for 1 <= top_k <= 8 it never enters the support; a slot
 * whose logits are all NaN then has an empty support: q_i all zero and
 * draft 0).  One CTA
 * (one warp when 1 <= top_k <= 8, V <= 1024, V % 4 == 0 and the three
 * float arrays are 16-byte aligned); V <= 8192, 1 <= gamma <= 64, T > 0. */
int evs_markov_draft(const float* trunk_logits_dev, const float* markov_dev, int32_t V, const int32_t* prev_dev,
                     const float* u_dev, int32_t gamma, float T, int32_t top_k, int32_t mode,
                     int32_t* drafts_dev, float* q_dev, cudaStream_t stream);

/* Commit ([abstract] (i): per-position state slicing with zero
 * recomputation).  keep in [0, n] tokens of the pending block are consumed:
 * FIR window <- ext rows [keep, keep+L-1); IIR state <- state after block
 * position keep-1 (keep = 0: unchanged); KV length, position += keep.
 * Bank flips only - no data is copied.  EVS_ERR_STATE without a pending
 * verify; EVS_ERR_ARG if keep is out of range. */
int evs_commit(evs_state* s, int32_t keep, cudaStream_t stream);
/* Same with keep = accepted_dev[0] + 1 read on the device (the output of
 * evs_accept), so a verify-accept-commit round needs no host round trip and
 * can be graph-captured.  A keep outside [0, n] sets EVS_DEV_BAD_KEEP and
 * leaves the state as before the verify. */
int evs_commit_dev(evs_state* s, const int32_t* accepted_dev, cudaStream_t stream);

/* One round as a single graph launch: verify(tokens) -> logits; probs (if
 * mode == EVS_SAMPLE) -> p; accept -> accepted, token; commit_dev.  p_dev
 * may be null in greedy mode. */
int evs_round(evs_state* s, const int32_t* tokens_dev, int32_t n, float* logits_dev,
              float* p_dev, const float* q_dev, const float* u_dev, float T, int32_t top_k,
              int32_t mode, int32_t* out_accepted_dev, int32_t* out_token_dev,
              cudaStream_t stream);
/* The same round with the block and the result in host memory (any host
 * buffers): copies tokens_host [n] in, runs the round (arguments as
 * evs_round; n <= 16), and returns once accepted_host[0] and token_host[0]
 * hold the result (the call synchronises the stream).  The two
 * copies go through the state's pinned staging and are part of the round's
 * graph, so a round costs one graph launch and one synchronisation. */
int evs_round_host(evs_state* s, const int32_t* tokens_host, int32_t n, float* logits_dev,
                   float* p_dev, const float* q_dev, const float* u_dev, float T, int32_t top_k,
                   int32_t mode, int32_t* accepted_host, int32_t* token_host, cudaStream_t stream);
/* Batched round ([systems] batched verification with ragged per-sequence
 * rollback, with the bookkeeping on the device): one graph launch doing
 * evs_verify_batch over the nseq sequences' blocks, then (EVS_SAMPLE) the
 * target distributions of all rows, the accept rule of every sequence and
 * every sequence's commit with its own keep = accepted + 1.  Row layout as
 * evs_verify_batch: sequence b owns rows r0 = sum of n_host[0..b-1] ..
 * r0 + n_host[b] - 1 of tokens_dev (pending token, then its drafts),
 * logits_dev and p_dev [sum n][V]; q_dev [sum n][V] (row r0 + i: the
 * drafter distribution of draft i + 1; the sequence's last row unused) and
 * u_dev [sum n] (rows r0 .. r0 + n_host[b] - 1: that sequence's uniforms)
 * in sample mode (p, q, u may be null in greedy mode).  Outputs
 * out_accepted_dev[b], out_token_dev[b].  Each sequence's results and state
 * equal those of its own evs_round bit for bit.  Limits and errors as
 * evs_verify_batch; V <= 8192. */
int evs_round_batch(evs_state* const* states_host, int32_t nseq, const int32_t* tokens_dev,
                    const int32_t* n_host, float* logits_dev, float* p_dev, const float* q_dev,
                    const float* u_dev, float T, int32_t top_k, int32_t mode,
                    int32_t* out_accepted_dev, int32_t* out_token_dev, cudaStream_t stream);

/* ---------------------------------------------------------------- operators
 * Single-operator entry points over caller-owned buffers: the same kernels
 * the model path runs, with the mixer input given as a plain matrix instead
 * of GEMM partial sums.  For operator-level parity and timing.            */

/* Hyena FIR mixer for one block ([systems], [prereq1]).
 * abv_dev [n][3d] storage dtype (a|b|v), taps [L][d], ring_dev
 * [L-1+n_max][d] float32 (the input of position p at row p mod (L-1+n_max),
 * the window being positions pos-L+1 .. pos-1; rows before position 0 must
 * be zero), book_dev: pos is read, nothing written.  Writes g_dev [n][d]
 * storage dtype = a * (h (*) (b*v)) and the block's inputs b*v at positions
 * pos .. pos+n-1 of the ring.  Needs d % 32 == 0 and 1 <= L <= 256. */
int evs_op_fir(int32_t L, int32_t d, int32_t n, int32_t n_max, int32_t dtype,
               const void* abv_dev, const float* taps_dev, float* ring_dev,
               const evs_book* book_dev, void* g_dev, cudaStream_t stream);
/* Hyena modal IIR mixer for one block.  State banks [n_max][d][M][2];
 * reads the state at (iir_bank, iir_slot), writes the n per-position states
 * to slots 0..n-1 of bank 1-iir_bank.  M must be a power of two <= 32 and
 * d * M a multiple of 256. */
int evs_op_iir(int32_t M, int32_t d, int32_t n, int32_t n_max, int32_t dtype,
               const void* abv_dev, const float* lambda_dev, const float* residue_dev,
               float* st0_dev, float* st1_dev, const evs_book* book_dev, void* g_dev,
               cudaStream_t stream);
/* Block-causal attention for one block: qkv_dev [n][3*H*Dh] (q|k|v, heads
 * contiguous) storage dtype; caches [H][ctx_max][Dh]; Dh in {32, 64, 128};
 * rotary embedding at positions pos..pos+n-1 (angle pos * base^(-2i/Dh)
 * reduced exactly in 64-bit fixed point, sin / cos in float),
 * k/v appended to the caches at those rows, query i attends rows
 * 0..pos+i (EvSpark discussion post, "What we implemented").  Writes g_dev
 * [n][H*Dh].  scratch: evs_op_attention_scratch_bytes, device memory the
 * call fills (rotary table, tensor maps of the caches, zeroed counters)
 * before its kernels, synchronously on the stream: not for stream capture.
 * bf16 caches with Dh 64 / 128 stream K and V by tensor-map copies (caches
 * 16-byte aligned); above 8192 positions one kernel also does the rotary
 * embedding, the append and the fold of the key splits. */
size_t evs_op_attention_scratch_bytes(int32_t H, int32_t Dh, int64_t ctx_max, int32_t chunk, int32_t n_max);
int evs_op_attention(int32_t H, int32_t Dh, int32_t n, int32_t n_max, int64_t ctx_max,
                     int32_t chunk, float rope_base, int32_t dtype, const void* qkv_dev,
                     void* k_cache_dev, void* v_cache_dev, evs_book* book_dev, void* g_dev,
                     void* scratch_dev, size_t scratch_bytes, cudaStream_t stream);
/* Commit on a bare book after an operator call on a block of n tokens:
 * keep in [0, n]; flips the FIR / IIR banks and advances pos as evs_commit
 * does. */
int evs_op_commit(evs_book* book_dev, int32_t keep, int32_t n, cudaStream_t stream);
/* Skinny GEMM Y[n][N] = X[n][K] W^T (weight-streaming path; tensor cores
 * for bf16).  W [N][K], X [n][K] storage dtype, n <= 16; Y float32.
 * scratch: evs_op_gemm_scratch_bytes.  Synchronizes stream once before the
 * launch (slot-table upload); the GEMM itself runs asynchronously.  The
 * int at byte offset evs_op_gemm_scratch_bytes(N, K, dtype) - 256 of
 * scratch is the launch's device status: zeroed before the launch, it holds
 * EVS_DEV_TIMEOUT afterwards if a bounded pipeline wait gave up (Y is then
 * incomplete); the caller reads it after the stream completes. */
size_t evs_op_gemm_scratch_bytes(int32_t N, int32_t K, int32_t dtype);
int evs_op_gemm(const void* w_dev, const void* x_dev, int32_t N, int32_t K, int32_t n,
                int32_t dtype, float* y_dev, void* scratch_dev, size_t scratch_bytes,
                cudaStream_t stream);
/* The same GEMM without caller scratch: an engineering entry point with no
 * counterpart in the pages.  Same arguments (minus the scratch), layout,
 * results and argument errors as evs_op_gemm, but it allocates no device
 * memory: its partial slots, slot table, arrival counters and error flag
 * live in one library-owned device array of EVS_OP_GEMM_STATIC_SCRATCH_BYTES
 * per device.
 * It serves callers that must not allocate on their path (a serving loop
 * that forbids allocation once running; a plug-in whose host framework owns
 * all device memory).  A shape whose scratch need (evs_op_gemm_scratch_bytes)
 * exceeds the array returns EVS_ERR_CAPACITY before any device work.  The
 * array's address is looked up on the first call on each device: make that
 * call outside stream capture.  Each call clears the counters and the error
 * flag with memsets and synchronizes `stream` after uploading the slot
 * table, as evs_op_gemm does.  Because the device status sits in the
 * library's array, the call also waits for the GEMM and reads the status
 * back (synchronous): a bounded pipeline wait that gave up returns
 * EVS_ERR_DEVICE (Y incomplete).  Calls share the array: calls that
 * overlap in time on one device (other streams or host threads) race, so
 * the caller serializes them. */
#define EVS_OP_GEMM_STATIC_SCRATCH_BYTES ((size_t)4 << 20)
int evs_op_gemm_static(const void* w_dev, const void* x_dev, int32_t N, int32_t K, int32_t n,
                       int32_t dtype, float* y_dev, cudaStream_t stream);

/* Self-test of the device-side bounded wait that guards every pipeline wait
 * of the GEMM (no counterpart in the pages): one thread waits on an
 * mbarrier nothing arrives on, for limit_ns in [1e3, 1e9]; the expiry ORs
 * EVS_DEV_TIMEOUT into *status_dev (device int, caller-owned) and the
 * kernel returns normally, leaving the context usable.  Asynchronous on
 * stream. */
int evs_selftest_wait_timeout(int32_t* status_dev, int64_t limit_ns, cudaStream_t stream);

/* ---------------------------------------------------------------- profiling */
/* Times every weight GEMM of one verify step of n tokens (per layer: in,
 * out, gate/up, down; then the head) with CUDA events around each launch,
 * on stream; synchronous.  A short fixed-length busy kernel runs ahead so
 * the events see only GPU time.  ms_host[i] = launch i's duration,
 * bytes_host[i] = its algorithmic bytes (weights + activations in +
 * outputs); *count = number of launches (4 * n_layers + 1 <= max_launches).
 * Each launch ends as in a verify step (partial slots left for the consumer
 * where the step does that, else the summed output; residual GEMMs write
 * their sums to scratch instead of the residual stream).  Uses the state's
 * workspaces; leaves the decoding state unchanged. */
int evs_profile_gemms(evs_state* s, int32_t n, float* ms_host, int64_t* bytes_host,
                      int32_t max_launches, int32_t* count, cudaStream_t stream);
/* The same GEMMs as they run in a verify step, back to back: one CUDA
 * graph of all 4 * n_layers + 1 launches with programmatic dependent launch
 * between them and each GEMM warming L2 with the next weight matrix's first
 * units (the step without its small kernels in between).  Three warm-up
 * launches of the graph, then reps (1..1000) timed with CUDA events on
 * stream; synchronous.  *ms_per_chain = average time of one chain,
 * *bytes_per_chain = its algorithmic bytes, *launches = GEMMs per chain.
 * Uses the state's workspaces; leaves the decoding state unchanged. */
int evs_profile_gemm_chain(evs_state* s, int32_t n, int32_t reps, float* ms_per_chain,
                           int64_t* bytes_per_chain, int32_t* launches, cudaStream_t stream);

/* ---------------------------------------------------------------- misc */
const char* evs_last_error(void);
const char* evs_version(void);
/* Number of kernels the library enqueued since load (all entry points). */
int64_t evs_kernel_launches(void);
/* Kernels one evs_verify_block(n) enqueues on this state (graph nodes). */
int32_t evs_verify_kernel_count(const evs_state* s, int32_t n);

#ifdef __cplusplus
}
#endif
#endif /* EVS_H */
