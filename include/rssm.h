/*
 * rssm.h — C ABI of the GB300 ReplaySSM hot path (gated delta rule, GDN and KDA).
 *
 * What the operations compute, restated from the pages they come from:
 *
 *  - LightLLM PR #1690 "feat: add ReplaySSM state modes for GDN and KDA"
 *    (PR description and commit messages): per request, a canonical checkpoint
 *    state plus a buffer of accepted-token records with a cursor; decode replays
 *    checkpoint + history + the new token; a ring that the next window would
 *    overflow is folded inside the decode kernel; the cursor advances once per
 *    step after the last layer; a restored slot has its cursor cleared; deltas
 *    are stored in fp32, keys in fp16 for bf16 activations.
 *  - SGLang fork PR jianc99/sglang#2 (GDN ReplaySSM for DFLASH/DSPARK), commit
 *    messages and "Modifications": speculative verify writes its T draft records
 *    at ring positions [write_pos, write_pos + T) and solves the window in the
 *    (I + A)^-1 triangular form with causal selects, so non-finite values at
 *    rejected drafts never reach accepted outputs; commit trims the rejected
 *    tail and (fold-every mode) folds the accepted window into the checkpoint;
 *    rows whose state slot is null (-1) are skipped by every kernel.
 *  - vLLM PR #64699 "[Feature][MRV2] Enable Qwen3.5 GDN ReplaySSM standard
 *    decode", commit messages: a per-row forced flush (fold) at any boundary.
 *
 * Per token t of a (request, value head) with state S[dk][dv]:
 *   GDN: S <- exp(g_t) S        KDA: S <- diag(exp(g_t)) S   (g_t per key channel)
 *   d_t = beta_t (v_t - S^T k_t);  S <- S + k_t d_t^T;  o_t = scale S^T q_t.
 * Value head h reads key head h / (HV/HK).
 *
 * Memory ownership: the caller allocates every device buffer and owns every
 * stream. The library borrows the pointers given to rssm_alloc for the life of
 * the handle and allocates nothing on the device; the handle itself is a small
 * host object. All index/length arrays passed per call are DEVICE pointers, so
 * no call synchronises the device or allocates (rssm_get_device_error excepted,
 * which synchronises the given stream). Every enqueueing call may be captured
 * in a CUDA graph.
 *
 * Errors: arguments the host can check are validated before anything is
 * enqueued; a failed check returns RSSM_ERR_INVALID_ARG or
 * RSSM_ERR_UNSUPPORTED and launches nothing. Conditions only the device can see
 * (a slot index >= n_slots, a cursor outside [0, L], an accepted length outside
 * [0, T]) set bits in the device error word and the affected row is skipped;
 * the kernels never trap. A null slot (-1) is not an error: its row is skipped
 * and its outputs are left untouched. Two live rows of one call must not name
 * the same slot (the result is then undefined). Launch failures return
 * RSSM_ERR_CUDA. No C++ exception crosses this ABI.
 *
 * Bounded waits: every wait of a kernel for its own async copies gives up
 * after 0.5 s and sets RSSM_DEVERR_TIMEOUT (a copy that never lands is a
 * hardware fault; nothing in normal operation comes near the limit). What the
 * affected row of a replay or fold launch then holds:
 *  - a wait for the window rows, or for the history records of a window that
 *    folds: nothing of the row is written (outputs, records, fold_out,
 *    checkpoint);
 *  - a later wait (the history of a window that does not fold, a checkpoint
 *    chunk): no output, delta, value or fold_out is written and no checkpoint
 *    chunk from the failed one on is stored back. A window that does not fold
 *    may have written its keys, gates and betas at ring positions [c, c + T),
 *    past the committed history (the row's committed state is untouched); a
 *    row that folds may have stored the chunks before the failed one already
 *    folded, so its checkpoint is then part old, part folded.
 * The cursor kernels do not see the failure (decode's advance_cursor, commit
 * and fold still move the cursor). A caller that finds the bit set must treat
 * the step as failed and restore the slots it touched (write a checkpoint,
 * rssm_reset_slots). Copies still in flight after a second bounded wait may
 * land after the CTA has left.
 *
 * Layouts (row-major, element counts; "tok" = r*T + i for row r, token i):
 *   q, k : [B*T][HK][dk]  in_dtype          v, o : [B*T][HV][dv] in_dtype
 *   beta : [B*T][HV] fp32                   g    : [B*T][HV] (GDN) | [B*T][HV][dk] (KDA) fp32
 *   state    : [n_layers][n_slots][HV][dk][dv]  state_dtype (the checkpoint)
 *   ring_k   : [n_layers][n_slots][HV][L][dk]   ring_k_dtype (one copy per value head)
 *   ring_d   : [n_layers][n_slots][HV][L][dv]   ring_d_dtype
 *   ring_g   : [n_layers][n_slots][HV][L]       (GDN) | [..][L][dk] (KDA) fp32
 *   ring_v   : [n_layers][n_slots][HV][L][dv]   in_dtype
 *   ring_beta: [n_layers][n_slots][HV][L]       fp32
 *   cursor   : [n_slots] int32, shared by all layers
 *   err_word : [1] uint32
 */
#ifndef RSSM_H_
#define RSSM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum rssm_status {
  RSSM_OK = 0,
  RSSM_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad index or size      */
  RSSM_ERR_UNSUPPORTED = 2,  /* valid but not built: dims, dtypes, smem limits  */
  RSSM_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed             */
  RSSM_ERR_DEVICE = 4        /* rssm_get_device_error found a non-zero word      */
} rssm_status;

enum { RSSM_ALGO_GDN = 0, RSSM_ALGO_KDA = 1 };
enum { RSSM_F32 = 0, RSSM_BF16 = 1, RSSM_F16 = 2 };

/* Activation of the short causal convolution (rssm_conv_window). */
enum { RSSM_CONV_ACT_NONE = 0, RSSM_CONV_ACT_SILU = 1 };
enum { RSSM_COMMIT_LAZY = 0, RSSM_COMMIT_FOLD_EVERY = 1 };

/* Kernel family serving rssm_decode / rssm_verify (rssm_set_plan). */
enum { RSSM_PLAN_AUTO = 0, RSSM_PLAN_ROWS = 1, RSSM_PLAN_PIPE = 2, RSSM_PLAN_TC = 3 };

/* Bits of the device error word. */
enum {
  RSSM_DEVERR_SLOT = 1u,     /* slot index >= n_slots                 */
  RSSM_DEVERR_CURSOR = 2u,   /* cursor outside [0, L]                 */
  RSSM_DEVERR_ACCEPT = 4u,   /* accepted length outside [0, T]        */
  RSSM_DEVERR_TIMEOUT = 8u,  /* a bounded wait on a tile copy ran out */
  RSSM_DEVERR_SEQLEN = 16u   /* ragged window offsets out of order or wider than max_T */
};

/*
 * Store configuration. Supported: dk, dv in {32, 64, 128}; HV a multiple of HK;
 * 1 <= max_T <= 16; max_T <= L <= 64 (a ring shorter than
 * the widest window is refused, SGLang fork PR jianc99/sglang#2, first commit;
 * a longer ring is RSSM_ERR_UNSUPPORTED: a fold carries the whole history and
 * the fold kernel takes at most 64 records);
 * in_dtype F32|BF16; state_dtype F32|BF16; ring_k_dtype F32|F16|BF16;
 * ring_d_dtype F32|F16. commit_mode selects what rssm_commit does.
 */
typedef struct rssm_config {
  int32_t algo;
  int32_t n_layers;
  int32_t n_slots;
  int32_t HK;
  int32_t HV;
  int32_t dk;
  int32_t dv;
  int32_t L;
  int32_t max_T;
  int32_t in_dtype;
  int32_t state_dtype;
  int32_t ring_k_dtype;
  int32_t ring_d_dtype;
  int32_t commit_mode;
  float scale;
} rssm_config;

/* Device buffers (layouts above). All must be non-null; state, ring_k, ring_d,
 * ring_g and ring_v must be 16-byte aligned (they move by bulk async copies).
 * Borrowed for the life of the handle. */
typedef struct rssm_buffers {
  void *state;
  void *ring_k;
  void *ring_d;
  float *ring_g;
  void *ring_v;
  float *ring_beta;
  int32_t *cursor;
  uint32_t *err_word;
} rssm_buffers;

/* Byte sizes of each buffer for a configuration. */
typedef struct rssm_sizes {
  size_t state;
  size_t ring_k;
  size_t ring_d;
  size_t ring_g;
  size_t ring_v;
  size_t ring_beta;
  size_t cursor;
  size_t err_word;
} rssm_sizes;

typedef struct rssm_handle rssm_handle;

/* Pure host: fills *out for a valid configuration. */
rssm_status rssm_required_bytes(const rssm_config *cfg, rssm_sizes *out);

/* Validates cfg and buffers, prepares kernel attributes on the current device
 * and returns a host handle in *out (freed by rssm_free). Does not touch the
 * buffers' contents: the caller zeroes cursor and err_word and writes the
 * initial checkpoint. */
rssm_status rssm_alloc(const rssm_config *cfg, const rssm_buffers *buf,
                       rssm_handle **out);
void rssm_free(rssm_handle *h);

/*
 * Width-1 replay decode of one layer (LightLLM PR #1690, commit messages on
 * decode and on the fused fold). For each row r with s = slot[r] >= 0:
 * c = cursor[s]; fold = force[r] || c + 1 > L. On fold the history is folded
 * into the checkpoint first (S0 <- replayed state) and the new record goes to
 * ring position 0, else to c. Writes o (B rows), the token's record
 * (k, d, g, v, beta; each value head keeps its own copy of the key) and, if
 * fold_out is non-null,
 * fold_out[r] = fold (0/1) for live rows. q, k, v (and g for KDA) must be
 * 16-byte aligned; beta, g (GDN) and slot 4-byte aligned. When advance_cursor is non-zero
 * (the last layer of the step) the cursor kernel then sets
 * cursor[s] = (fold ? 0 : c) + 1. force and fold_out may be null.
 * B == 0 is a no-op. Pointers are device pointers; stream is a cudaStream_t.
 */
rssm_status rssm_decode(rssm_handle *h, int32_t layer, const void *q,
                        const void *k, const void *v, const float *beta,
                        const float *g, const int32_t *slot,
                        const uint8_t *force, int32_t B, void *o,
                        uint8_t *fold_out, int32_t advance_cursor,
                        void *stream);

/*
 * Speculative verify of one layer: a window of T (1 <= T <= max_T) draft tokens
 * per row, same rules as decode with c + T > L as the overflow test; writes
 * T outputs per row and the T records at [base, base + T). Never moves the
 * cursor (rssm_commit does). Non-finite inputs at positions the later commit
 * rejects cannot change accepted outputs, accepted records or the state.
 */
rssm_status rssm_verify(rssm_handle *h, int32_t layer, const void *q,
                        const void *k, const void *v, const float *beta,
                        const float *g, const int32_t *slot,
                        const uint8_t *force, int32_t B, int32_t T, void *o,
                        uint8_t *fold_out, void *stream);

/*
 * Ragged speculative verify of one layer: windows of different lengths packed
 * into one token list (LightLLM PR #1690, commit messages: request windows
 * read from cu_seqlens over [tokens, heads, dim] inputs; SGLang fork PR
 * jianc99/sglang#2, "Related upstream work": verify on packed ragged tokens).
 * cu_seqlens is a device int32[B + 1]; row r's window is tokens
 * [cu_seqlens[r], cu_seqlens[r+1]) of q, k [N, HK, dk], v [N, HV, dv],
 * beta [N, HV], g [N, HV] (GDN) or [N, HV, dk] (KDA) and o [N, HV, dv], with
 * N = cu_seqlens[B]. Per row the rules of rssm_verify hold with T_r =
 * cu_seqlens[r+1] - cu_seqlens[r] in place of T (fold = force[r] ||
 * c + T_r > L). A row with T_r == 0 is idle: nothing is read or written for
 * it, fold_out[r] is left as it is. max_T (1 <= max_T <= the configuration's
 * max_T) bounds every T_r and picks the kernel width; a row whose offsets
 * are negative, decreasing or wider than max_T sets RSSM_DEVERR_SEQLEN and is
 * skipped. cu_seqlens must be 4-byte aligned; other alignment and error
 * rules as rssm_verify. Per-row forced folds (force) cover a caller that
 * must hold the exact state at its own block boundaries (vLLM PR #64699,
 * commit messages on align mode).
 */
rssm_status rssm_verify_ragged(rssm_handle *h, int32_t layer, const void *q,
                               const void *k, const void *v,
                               const float *beta, const float *g,
                               const int32_t *cu_seqlens,
                               const int32_t *slot, const uint8_t *force,
                               int32_t B, int32_t max_T, void *o,
                               uint8_t *fold_out, void *stream);

/*
 * Replay prefill of one layer (LightLLM PR #1690, commit messages: prefill
 * writes the canonical state directly and leaves the cursor at zero). Row r's
 * prompt is tokens [cu_seqlens[r], cu_seqlens[r+1]) of q, k [N, HK, dk],
 * v [N, HV, dv], beta [N, HV], g [N, HV] (GDN) or [N, HV, dk] (KDA), any
 * length >= 0. For each row with s = slot[r] >= 0 and at least one token, the
 * prompt runs through the gated delta rule from the row's committed state
 * (checkpoint plus its c = cursor[s] ring records), o [N, HV, dv] (input
 * dtype) takes every token's output, and the checkpoint of (layer, s) takes
 * the final state (rounded to the state dtype); the ring is not written. When
 * reset_cursor is non-zero (the last layer of the step) the cursor of every
 * such row is then set to 0, so every layer reads the same history before.
 * Rows with a null slot or no tokens are left untouched (outputs included).
 * cu_seqlens is a device int32[B + 1], 4-byte aligned; offsets that are
 * negative or decreasing set RSSM_DEVERR_SEQLEN and skip the row. Input
 * alignment and other error rules as rssm_decode.
 */
rssm_status rssm_prefill(rssm_handle *h, int32_t layer, const void *q,
                         const void *k, const void *v, const float *beta,
                         const float *g, const int32_t *cu_seqlens,
                         const int32_t *slot, int32_t B, void *o,
                         int32_t reset_cursor, void *stream);

/*
 * Native fused-recurrent decode of one layer, the path ReplaySSM replaces
 * (LightLLM PR #1690, PR description: the native mode writes the recurrent
 * state back every step). It is here as a comparison point: for each row r
 * with s = slot[r] >= 0 it treats the layer's checkpoint of (s, h) as the live
 * state and applies one token, S <- decay(g) S; d = beta (v - S^T k);
 * S <- S + k d^T; o = scale S^T q, storing S back (rounded to the state dtype)
 * and writing o (B rows, input dtype). The ring and the cursor are neither
 * read nor written, so mixing it with rssm_decode on the same slots is only
 * meaningful while their rings are empty. Same input layout, alignment and
 * error rules as rssm_decode; null slots are skipped.
 */
rssm_status rssm_native_decode(rssm_handle *h, int32_t layer, const void *q,
                               const void *k, const void *v, const float *beta,
                               const float *g, const int32_t *slot, int32_t B,
                               void *o, void *stream);

/*
 * Commit the last verify of every layer (SGLang fork PR jianc99/sglang#2,
 * fourth commit). accept_len[r] in [0, T]; slot/force/T must equal the
 * verify's. LAZY: cursor[s] = base + a (rejected tail trimmed). FOLD_EVERY:
 * for every layer S0 <- fold of the base + a records, then cursor[s] = 0.
 */
rssm_status rssm_commit(rssm_handle *h, const int32_t *slot,
                        const uint8_t *force, const int32_t *accept_len,
                        int32_t B, int32_t T, void *stream);

/*
 * Commit the last ragged verify of every layer: as rssm_commit with T_r =
 * cu_seqlens[r+1] - cu_seqlens[r] per row and accept_len[r] in [0, T_r];
 * slot, force, cu_seqlens and max_T must equal the verify's. Idle rows
 * (T_r == 0) keep their cursor and checkpoint.
 */
rssm_status rssm_commit_ragged(rssm_handle *h, const int32_t *slot,
                               const uint8_t *force, const int32_t *accept_len,
                               const int32_t *cu_seqlens, int32_t B,
                               int32_t max_T, void *stream);

/*
 * Conv-state window of a layer's short causal convolution, the second
 * per-request state beside the SSM (LightLLM PR #1690, commit messages: page
 * save, PD and DP copy the accepted conv window; SGLang fork PR
 * jianc99/sglang#2, fifth commit: the ring commit rolls the conv back). The
 * pages do not print the convolution; it is read as depthwise and causal of
 * width K: per live row r (slot[r] >= 0) and channel c,
 *     y_t[c] = act(bias[c] + sum_{i<K} w[c][i] * xp[t + i][c]),
 *     xp = [window[s] (K-1 rows), x_{r,0}, ..., x_{r,T-1}],
 * act = identity (RSSM_CONV_ACT_NONE) or SiLU (RSSM_CONV_ACT_SILU).
 * Layouts (device pointers, no alignment beyond the element size):
 * x, y [B*T][D] and window [n_slots][K-1][D] in dtype (RSSM_F32 or RSSM_BF16),
 * draft [n_slots][T][D] in dtype, w [D][K] fp32, bias [D] fp32 or null.
 * With commit_now (decode) the window moves on by the T tokens at once and
 * draft is not used (may be null); otherwise the window is left as it is and
 * the T inputs are kept in draft[s] for rssm_conv_commit. 2 <= K <= 8. Null
 * rows are skipped; a slot >= n_slots sets RSSM_DEVERR_SLOT in err_word (may
 * be null) and skips the row. The caller owns every buffer; nothing is
 * allocated and the call is capturable.
 */
rssm_status rssm_conv_window(const void *x, const float *w, const float *bias,
                             void *window, void *draft, const int32_t *slot,
                             int32_t B, int32_t T, int32_t D, int32_t K,
                             int32_t n_slots, int32_t dtype, int32_t act,
                             int32_t commit_now, void *y, uint32_t *err_word,
                             void *stream);

/*
 * Conv rollback on commit: window[s] <- the last K-1 rows of
 * [window[s], draft[s][0 .. a)], a = accept_len[r] in [0, T] (outside:
 * RSSM_DEVERR_ACCEPT, row skipped). T, D, K, dtype and the slots must be those
 * of the rssm_conv_window call that filled draft.
 */
rssm_status rssm_conv_commit(void *window, const void *draft,
                             const int32_t *slot, const int32_t *accept_len,
                             int32_t B, int32_t T, int32_t D, int32_t K,
                             int32_t n_slots, int32_t dtype, uint32_t *err_word,
                             void *stream);

/* Explicit fold of every layer's history into its checkpoint, then cursor <- 0
 * (LightLLM PR #1690: materialise the canonical state). */
rssm_status rssm_fold(rssm_handle *h, const int32_t *slot, int32_t B,
                      void *stream);

/* Restore semantics: cursor <- 0 for the given slots, so a slot whose
 * checkpoint was just written (state copy, restore) starts with an empty
 * history (LightLLM PR #1690, PR description and commit messages). */
rssm_status rssm_reset_slots(rssm_handle *h, const int32_t *slot, int32_t B,
                             void *stream);

/* Synchronises `stream`, reads the device error word into *out and clears it
 * when `clear` is non-zero. Returns RSSM_ERR_DEVICE if the word was non-zero.
 * For tests and debugging; not capturable. */
rssm_status rssm_get_device_error(rssm_handle *h, uint32_t *out, int32_t clear,
                                  void *stream);

/*
 * Which kernel serves rssm_decode and rssm_verify of this handle. Both compute
 * the same replay (same inputs, outputs, records and fold decisions; sums may
 * differ in rounding order):
 *  - RSSM_PLAN_ROWS: one CTA per (request row, value head) for the launch;
 *  - RSSM_PLAN_PIPE: the pipelined kernel, one persistent CTA per SM walking
 *    the (row, value head) items, checkpoint chunks streamed continuously
 *    across items while other warps prepare the next item and solve the last.
 *    A bounded wait that runs out there stops the CTA: the rows of the items
 *    it had not finished are left untouched (as above for the item in
 *    progress).
 *    It serves GDN stores with dk = dv = 128, L <= 16 and L a multiple of 4,
 *    fp32 or fp16 deltas, calls with T <= 8 and B <= 512 (uniform windows);
 *    calls outside that run on the per-row kernel.
 *  - RSSM_PLAN_TC: the per-row kernel, whose GDN windows of 3..8 tokens
 *    (uniform, not ragged) stream the checkpoint tile through the
 *    5th-generation tensor cores (tcgen05 MMAs, tensor-memory accumulators;
 *    fp32 operands as tf32 hi + lo pairs, so the products keep fp32
 *    accuracy); a fold of up to 16 records runs there too. The folds of
 *    rssm_commit (fold-every stores) and rssm_fold compute their rank-n
 *    update on the tensor cores as well when L <= 32. It serves GDN stores
 *    with dv = 128 and dk a multiple of 32; other calls of such a store run
 *    as RSSM_PLAN_ROWS.
 *  - RSSM_PLAN_AUTO (after rssm_alloc): the per-row kernel.
 * RSSM_PLAN_PIPE or RSSM_PLAN_TC on a store it cannot serve returns
 * RSSM_ERR_UNSUPPORTED. Host
 * state only; takes effect at the next launch.
 */
rssm_status rssm_set_plan(rssm_handle *h, int32_t plan);

/*
 * Test and debugging hook of the bounded waits (no counterpart in the pages:
 * it exists so that the timeout path above can be exercised without a fault).
 * barrier: -1 turns the hook off (the state after rssm_alloc); 0 the window
 * rows' barrier, 1 the history records', 2 + j that of checkpoint chunk j of
 * the launch's first item (every row for the per-row kernel). While the hook
 * is on, every replay and fold launch of this handle leaves that barrier short
 * of what its copies bring, so every wait on it runs out after the usual
 * 0.5 s; the copies themselves all land. Host state only: takes effect at the
 * next launch. Never on in production calls.
 */
rssm_status rssm_debug_withhold(rssm_handle *h, int32_t barrier);

const char *rssm_status_string(rssm_status s);

/* ABI version of this header: 1. */
int32_t rssm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* RSSM_H_ */
