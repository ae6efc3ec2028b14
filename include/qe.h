/*
 * qe.h -- C ABI of the tiered (BF16 / INT2 / evicted) KV-cache decode path.
 *
 * The cache keeps, per (batch element, layer, KV head) "unit", a sink prefix
 * and the recent tokens in bf16, the top-Kf windows of w tokens in bf16, the
 * next Kq windows as 2-bit codes with float32 min/scale parameters, and
 * drops the rest.  Each decode step attends over that mixed set and adds
 * every window's attention mass (summed over the unit's GQA query heads) to
 * the window's cumulative score; every Omega steps the windows are
 * re-ranked and promoted, demoted or evicted.
 *
 * Sources (page title, section / equation):
 *  - QEvict reading notes (zhongzhuzhou.org, 2026-08-08): §2 Figure 1 (pipeline,
 *    windows start in full precision), §4.1 eq. "attention" and eq. "budget",
 *    §4.2 eq. (1) cumulative window score, §4.3 eq. (3) capacities, §4.4
 *    eqs. (4)-(6) and Algorithm 1 (routing, quantize-once ledger, promotion).
 *  - H2O: keeping heavy hitters by cumulative attention (PaperTrace 3.1.2):
 *    §2.1 step order, §5.1 GQA group sum and state arrays, §5.1 ties broken on
 *    the original position, §3.1 / §5.1 float32 score storage.
 *  - HqeKV reading notes (zhongzhuzhou.org, 2026-08-26): §2.3 eq. (2) uniform
 *    min/scale quantizer.
 *  - KV Cache technology evolution (zane-jiang.github.io): §5 KIVI axes (keys
 *    per channel across tokens, values per token).
 *
 * Conventions for every call:
 *  - All work is enqueued on the CUDA stream given to qe_init (the handle's
 *    stream) and returns without waiting, except where stated.  Device buffers
 *    passed in must stay valid until the stream has reached the call.
 *  - Status codes are returned, never exceptions or traps.  A device-side
 *    consistency flag (free-list underflow, table corruption, bounded wait
 *    expiry) is sticky; qe_synchronize() reports it as QE_ERR_DEVICE.
 *  - qe_last_error() returns a message for the last failing call on the
 *    handle (or on qe_init when the handle is NULL); the string is owned by the
 *    library and valid until the next call on that handle.
 *  - Unit index u = b * n_kv_heads + kvh; query head h of unit u is
 *    kvh * G + i, i < G = n_q_heads / n_kv_heads.
 *  - Window j of a sequence covers positions [j w, (j+1) w); the sink
 *    positions [0, n_sink) are carved out of window 0.
 */
#ifndef QE_H
#define QE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct qe_handle_s* qe_handle;

typedef enum {
  QE_OK = 0,
  QE_ERR_INVALID_ARG = 1,  /* bad pointer, index, size or unsupported shape */
  QE_ERR_OOM = 2,          /* device or pinned host allocation failed */
  QE_ERR_CAPACITY = 3,     /* appending beyond max_context, or a pool would overflow */
  QE_ERR_CUDA = 4,         /* a CUDA runtime call failed (message has the CUDA error string) */
  QE_ERR_TIMEOUT = 5,      /* a bounded device wait expired */
  QE_ERR_STATE = 6,        /* call not valid in the handle's current state */
  QE_ERR_HOST_STORE = 7,   /* pinned host backing store could not be mapped */
  QE_ERR_DEVICE = 8        /* sticky device-side consistency flag was raised */
} qe_status;

/* Tier of a window (qe_get_tiers). */
enum {
  QE_TIER_NONE = 0,      /* window not reached yet */
  QE_TIER_PINNED = 1,    /* bf16, not yet ranked (recent or awaiting its first routing event) */
  QE_TIER_FULL = 2,      /* bf16, among the top Kf */
  QE_TIER_QUANT = 3,     /* 2-bit codes + float32 min/scale, among the next Kq */
  QE_TIER_EVICTED = 4    /* dropped for good */
};

/* Capacity rule (QEvict notes §4.3 eq. (3); the mapping from the workloads'
 * token shares to window counts is this library's reading):
 *   0: Kf = kf, Kq = kq windows;
 *   1: Kf = max(0, floor((frac_bf16 L - n_sink - n_recent) / w)),
 *      Kq = floor(frac_int2 L / w);
 *   2: Kf as in 1, Kq = floor((budget_frac - frac_bf16) L * 4 d / M_q(w)),
 *      M_q(w) = w d / 2 + 8 d + 8 w bytes (codes + float32 min/scale).
 * L is the sequence length at the routing event; all in double precision. */
typedef struct {
  int batch;
  int n_layers;
  int n_q_heads;
  int n_kv_heads;      /* n_q_heads / n_kv_heads in {1, 2, 4} */
  int head_dim;        /* 64 or 128 */
  int window;          /* w: 16, 32 or 64 tokens */
  int route_period;    /* Omega (the caller calls qe_route every Omega steps) */
  int n_sink;          /* 0 <= n_sink < min(window, 16) */
  int n_recent;        /* recent region length, tokens, >= 1 */
  int max_context;     /* most tokens per sequence the cache will hold */
  int cap_mode;        /* 0, 1 or 2, see above */
  int kf, kq;          /* cap_mode 0 */
  double frac_bf16;    /* cap_mode 1, 2 */
  double frac_int2;    /* cap_mode 1 */
  double budget_frac;  /* cap_mode 2 */
  int out_fp32;        /* 1: qe_decode_step writes float32, 0: bf16 */
  /* Tiering (QE_TIERING_*).  QE_TIERING_TOKENS is the five-tier per-token cache of the HqeKV
   * reading notes (§3.1): every token is BF16, 4-bit or 2-bit uniform (eq. (2), per-token
   * min/scale for its key and its value), 1-bit normal (eqs. (3)-(4): per-token mean and
   * population std, centers +-Phi^-1(3/4), code 1 when x > mean) or evicted.  qe_route then
   * re-ranks (§3.5): the n_sink first and n_recent last tokens stay BF16; the others are
   * ranked by score (descending, ties to the lower position) and the ranks give the tiers in
   * the order BF16, 4-bit, 2-bit, 1-bit, evicted with counts
   *   max(0, floor(frac_bf16 L) - n_sink - n_recent), floor(frac_int4 L),
   *   floor(frac_int2 L), floor(frac_nq1 L), the rest
   * (double precision); a token only moves down (a token whose rank asks for a higher tier
   * keeps its own), and a token that moves is re-quantized from what its tier held (one
   * float32 fma per value).  Scores add each token's attention mass summed over the KV head's
   * query heads, on the last score_window decode steps before a re-rank (0: every step), and
   * restart at 0 after it when score_window > 0.  window, cap_mode, kf, kq and budget_frac are
   * unused; route_period is the re-rank period. */
  int tiering;
  double frac_int4;
  double frac_nq1;
  int score_window;
  /* Keys stored pre-RoPE (window tiering; QEvict notes §4.4: keys are quantized before the
   * rotary embedding and rotated again at their original positions).  rope_theta > 0: the
   * K passed to qe_append is pre-RoPE and every cached key (bf16, or dequantized 2-bit) is
   * rotated at its original position p before q . k: channel pairs (2i, 2i + 1) by the angle
   * p * rope_theta^(-2i / head_dim).  q is passed already rotated at its own position.
   * 0: keys are used as stored. */
  double rope_theta;
  /* 2-bit window slots beyond the most Kq at max_context (window tiering).  A freed slot keeps
   * its window's codes until it is handed out again (oldest first): a window demoted again by
   * then takes its codes back, and a kept window's codes are written to the host ledger only
   * when their slot is about to be handed to another window.  0: max(16, Kq / 2); -1: none;
   * n > 0: n slots. */
  int int2_slack;
} qe_config;

enum { QE_TIERING_WINDOWS = 0, QE_TIERING_TOKENS = 1 };

/* Token tiers of the five-tier mode (qe_get_token_tiers). */
enum {
  QE_TOK_BF16 = 0, QE_TOK_INT4 = 1, QE_TOK_INT2 = 2, QE_TOK_NQ1 = 3, QE_TOK_EVICTED = 4,
  QE_TOK_ABSENT = 255    /* position not appended yet */
};

/* Pointer-location flags for qe_append / qe_decode_step. */
enum {
  QE_DEVICE_PTRS = 0,  /* all buffers are device memory */
  QE_HOST_PTRS = 1     /* all buffers are host memory.  Page-locked, device-mapped buffers
                          (cudaHostAlloc, or registered as mapped) stay asynchronous: a
                          single-token append's K and V are read, and decode outputs written,
                          by the kernels in place over the host link; queries and multi-token
                          appends are copied in.  Pageable buffers are copied both ways, and
                          the copies then block the calling thread. */
};

/* Create a cache for cfg on the current CUDA device.  Allocates the device
 * window pools (bf16 slots for every window up to max_context, 2-bit slots for
 * the largest Kq), the window table and scores, and a pinned, device-mapped
 * host backing store that keeps the exact bf16 copy of every kept (Full or
 * Quantized) window, written when the window is first kept, and the 2-bit
 * ledger entry of every window that has been demoted and not evicted.
 * cuda_stream: a cudaStream_t (NULL = legacy default stream).  The handle
 * owns everything it allocates.  No kernel runs. */
qe_status qe_init(const qe_config* cfg, void* cuda_stream, qe_handle* out);

/* Free everything the handle owns (waits for its stream first). */
qe_status qe_destroy(qe_handle h);

const char* qe_last_error(qe_handle h);

/* Append n_tokens positions to every sequence of one layer.
 * k, v: [batch][n_kv_heads][n_tokens][head_dim] bf16 (row-major).
 * Windows reached for the first time start Pinned with score 0 (QEvict notes
 * §2 Figure 1: every window starts in full precision).  Prefill is one call
 * with n_tokens = prompt length; a decode step appends 1 token.
 * A single-token append launches nothing: the next qe_decode_step of the layer
 * writes the token inside its attention launch (any other call on the layer
 * writes it first).  Device and pinned host k and v must therefore stay valid
 * and unchanged until the stream reaches that call; pageable host k and v are
 * copied to the layer's own staging buffers at once.
 * Errors: QE_ERR_CAPACITY if the length would pass max_context. */
qe_status qe_append(qe_handle h, int layer, const void* k, const void* v, int n_tokens, int flags);

/* One decode step of one layer (QEvict notes §4.1 eq. "attention"; H2O page
 * §2.1 order: the token appended last is attended too).
 * Any finite bf16 keys, values and queries are served: 2-bit windows whose parameters, with
 * the step's queries, would push the tensor-core operands out of the f16 range take bf16
 * operands instead (decided per window from magnitudes recorded when it was packed), and keys
 * stored pre-RoPE always meet the queries in tf32.
 * q:   [batch][n_q_heads][head_dim] bf16.
 * out: [batch][n_q_heads][head_dim] float32 (out_fp32) or bf16.
 * Computes softmax(q K_acc^T / sqrt(d)) V_acc over the sink, the Pinned and
 * Full bf16 windows and the dequantized INT2 windows (x = code * s + z), and
 * adds each window's mass, summed over the unit's query heads, to its
 * float32 score (eq. (1) with the GQA group sum).  Sink tokens are never
 * scored.  A pinned host out is written by the combine kernel in place and
 * is complete once the stream has passed the call. */
qe_status qe_decode_step(qe_handle h, int layer, const void* q, void* out, int flags);

/* Routing event of one layer (layer = -1: all layers), QEvict notes §4.4
 * Algorithm 1: candidates = Full u Quantized u Pinned windows that are
 * complete and wholly older than the last n_recent positions (eq. (4));
 * sorted by score descending, ties to the lower window index (original
 * position); top Kf -> Full, next Kq -> Quantized, rest -> Evicted (eq. (5)).
 * A window quantized for the first time is packed from its bf16 values (keys
 * per channel over the window's tokens, values per token over head_dim,
 * eq. (2) with b = 2, round half to even, float32 min and scale).  A kept
 * window's exact bf16 values are in the host backing store; its codes stay in
 * its 2-bit slot after a promotion and are written to the store only when that
 * slot is handed to another window (int2_slack).  A later demotion reuses the
 * codes (from the old slot, else the store); a promotion takes back its old
 * bf16 slot when no window has reused it, else copies the stored values back.
 * layer = -1 checks every layer first (nothing is routed if one fails) and
 * routes all of them with one launch of each kernel.  All moves complete on
 * the handle's stream before it runs anything else. */
qe_status qe_route(qe_handle h, int layer);

/* ---------------------------------------------------------------- speculative verify
 * (window tiering; H2O page §5, speculative decoding: each draft query adds attention mass to
 * older positions, so a rejected draft's score increments must be rolled back; here they are
 * held aside and only the accepted ones are added).
 *
 * qe_verify appends n_q draft tokens and runs draft query j over the cache and drafts 0..j, as
 * n_q decode steps would, except that each query's window masses are kept per query instead of
 * being added to the scores.  Two paths compute it (the same results up to float32 summation
 * order):
 *  - fused (keys used as stored, n_q * group <= 64, n_q >= 5 by default): the drafts are
 *    appended in one launch and one attention launch reads every window of the cache once for
 *    all n_q * group query rows, on the tensor cores (tcgen05.mma, float32 accumulators in
 *    tensor memory; bf16 operands, a 2-bit window's dequantized keys as three exact bf16 parts,
 *    the probabilities as two bf16 parts, about 17 significant bits); a combine launch writes
 *    the outputs and each draft's window masses;
 *  - draft by draft (keys stored pre-RoPE, more rows, or fewer drafts): one append and one
 *    decode-step attention per draft.
 * qe_debug_inject(QE_DEBUG_VERIFY_PATH) overrides the choice.
 *   q:   [n_q][batch][n_q_heads][head_dim] bf16 (draft-major: draft j's queries are contiguous)
 *   k,v: [n_q][batch][n_kv_heads][head_dim] bf16
 *   out: [n_q][batch][n_q_heads][head_dim] float32 (out_fp32) or bf16
 * The layer then awaits qe_verify_commit; qe_append, qe_decode_step and qe_route on it fail
 * with QE_ERR_STATE until then.  Pointer rules and flags as for qe_append / qe_decode_step.
 * Errors: QE_ERR_INVALID_ARG (n_q outside 1..QE_VERIFY_MAX), QE_ERR_CAPACITY, QE_ERR_STATE. */
#define QE_VERIFY_MAX 16
qe_status qe_verify(qe_handle h, int layer, const void* q, const void* k, const void* v, void* out, int n_q,
                    int flags);

/* Keep drafts 0..n_accept-1 of the pending verify (0 <= n_accept <= n_q): the length becomes
 * L0 + n_accept, windows opened by rejected drafts close (their slots return to the free
 * list), and the accepted queries' window masses are added to the scores in draft order
 * (float32, as n_accept decode steps would have added them).  Stream-ordered. */
qe_status qe_verify_commit(qe_handle h, int layer, int n_accept);

/* Wait for the handle's stream and report the sticky device flag. */
qe_status qe_synchronize(qe_handle h);

/* ---------------------------------------------------------------- introspection */

typedef struct {
  int length;             /* tokens per sequence */
  int n_windows;          /* windows reached, ceil(length / w) */
  int routed_upto;        /* windows [0, routed_upto) have entered the candidate pool */
  int n_full, n_quant;    /* per unit */
  int n_pinned;           /* per unit, bf16 windows not yet ranked */
  int kf, kq;             /* capacities at the last routing event */
  int max_windows;        /* row length of qe_get_tiers / qe_get_scores */
  int units;              /* batch * n_kv_heads */
  double attn_bytes;      /* algorithmic bytes one qe_decode_step of this layer reads:
                             bf16 tokens * 4 d + INT2 windows * M_q(w) */
} qe_layer_info;

qe_status qe_get_layer_info(qe_handle h, int layer, qe_layer_info* info);

/* Tiers [units][max_windows] uint8 (QE_TIER_*); synchronous. */
qe_status qe_get_tiers(qe_handle h, int layer, uint8_t* host, size_t bytes);

/* Scores [units][max_windows] float32; synchronous. */
qe_status qe_get_scores(qe_handle h, int layer, float* host, size_t bytes);

/* Overwrite scores [units][max_windows] float32 (tests drive the router with
 * chosen scores); synchronous with respect to the host buffer. */
qe_status qe_set_scores(qe_handle h, int layer, const float* host, size_t bytes);

/* Contents of one Quantized window in canonical order; synchronous.
 * k_codes, v_codes: [w][head_dim] uint8 in 0..3 (rows below n_sink of window 0
 * are 0); k_min, k_scale: [head_dim] float32; v_min, v_scale: [w] float32.
 * Errors: QE_ERR_STATE if the window is not Quantized. */
qe_status qe_get_quant_window(qe_handle h, int layer, int unit, int window,
                              uint8_t* k_codes, uint8_t* v_codes,
                              float* k_min, float* k_scale, float* v_min, float* v_scale);

/* bf16 contents [w][head_dim] of a Pinned or Full window (or of the sink when
 * window = -1); synchronous. */
qe_status qe_get_bf16_window(qe_handle h, int layer, int unit, int window, uint16_t* k, uint16_t* v);

typedef struct {
  long long routes;        /* routing events run on this layer */
  long long first_packs;   /* windows quantized for the first time */
  long long ledger_reuses; /* demotions that reused stored codes */
  long long promotions;    /* Quantized -> Full */
  long long evictions;
  long long bf16_reclaims; /* promotions that took back their previous bf16 slot, whose
                              contents no other window had overwritten (no host read) */
  long long int2_reclaims; /* re-demotions that took back their previous 2-bit slot (no
                              host read of the ledger) */
  long long ledger_writes; /* ledgers written to the host store: a window's codes are saved
                              only when the 2-bit slot still holding them is handed to another
                              window while the window is kept */
} qe_route_stats;

/* Cumulative routing counters of one layer (layer = -1: summed); synchronous. */
qe_status qe_get_route_stats(qe_handle h, int layer, qe_route_stats* out);

/* One unit's record of the layer's latest routing event (diagnostics; QEvict reading notes §3
 * define selection churn as the Jaccard distance between the kept sets of consecutive routing
 * events, H2O page §5.1 the cutoff margin as the lowest kept score minus the highest dropped
 * one).  "Old" is the tier map before the event; windows entering the candidate pool from
 * Pinned are in no old set.  A cut score is -1 when that side of the cut is empty. */
typedef struct {
  int kf, kq;            /* capacities at the event */
  int full_old, full_new, full_both;   /* |F|, |F'|, |F and F'| (Full sets) */
  int kept_old, kept_new, kept_both;   /* the same for Full or Quantized */
  int promotions;        /* Quantized -> Full */
  int demotions;         /* Full -> Quantized */
  int evictions;         /* -> Evicted */
  float full_cut_kept;   /* score of the candidate ranked K_f (the lowest Full one) */
  float full_cut_next;   /* score of the candidate ranked K_f + 1 */
  float kept_cut_kept;   /* score of the candidate ranked K_f + K_q (the lowest kept one) */
  float kept_cut_next;   /* score of the candidate ranked K_f + K_q + 1 */
} qe_route_diag;

/* Copy the records of the layer's latest routing event for units [0, n_units) (unit = batch
 * element x KV head, in that order) into out; synchronous.  Records of a layer that has not
 * been routed are zero. */
qe_status qe_get_route_diag(qe_handle h, int layer, qe_route_diag* out, size_t n_units);

/* Profiling: qe_init, qe_append, qe_decode_step, qe_decode_step_noalloc, qe_verify,
 * qe_verify_commit, qe_route and qe_synchronize each open an NVTX range named after the call
 * (NVTX v3, header-only; without a profiler attached a range costs one test of a null
 * function pointer).  The ranges mark host-side enqueueing, not device time. */

/* Time every attention launch with CUDA events on the handle's stream (enable = 1) or stop
 * (0): the decode step's (qe_decode_step, and qe_verify draft by draft) and the fused verify's
 * (qe_verify with the tensor-core path; its combine launch is not timed).  qe_get_timing
 * returns the summed device time in ms, the number of launches and the summed algorithmic
 * bytes (the kept windows each launch reads) of the timed launches since the last enable, and
 * resets nothing. */
qe_status qe_set_timing(qe_handle h, int enable);
qe_status qe_get_timing(qe_handle h, double* attn_ms, long long* launches, double* attn_bytes);

/* Measurement aid: the mean CUDA-event time, in microseconds, of n launches (1 <= n <= 10000)
 * that have the window path's attention launch shape (its grid, block and dynamic shared memory,
 * programmatic serialization) and do nothing, enqueued back to back, each between two events
 * on the handle's stream.  That is the part of a timed attention launch that is launch and
 * event overhead rather than kernel work.  Synchronous; enqueues nothing that changes the
 * handle's state.  QE_ERR_STATE on a five-tier handle; QE_ERR_INVALID_ARG for n out of range
 * or a null us. */
qe_status qe_launch_overhead(qe_handle h, int n, double* us);

/* ---------------------------------------------------------------- five-tier introspection
 * (QE_TIERING_TOKENS handles; all synchronous; QE_ERR_STATE on a window-tiered handle) */

/* Tier of every position [units][max_context] uint8 (QE_TOK_*). */
qe_status qe_get_token_tiers(qe_handle h, int layer, uint8_t* host, size_t bytes);

/* Score of every position [units][max_context] float32 (0 for evicted and absent ones). */
qe_status qe_get_token_scores(qe_handle h, int layer, float* host, size_t bytes);

/* Tokens per unit [units][5] int32: ranked BF16, 4-bit, 2-bit, 1-bit, and the BF16 tail
 * (sink, recent and the tokens appended since the last re-rank). */
qe_status qe_get_token_counts(qe_handle h, int layer, int* host, size_t bytes);

/* One token: *tier (QE_TOK_*); for BF16 its key and value bf16 bits [head_dim] each; for a
 * quantized tier its codes [head_dim] each and params = {key p0, key p1, value p0, value p1}
 * (min and scale, or mean and std for the 1-bit tier).  Pointers of the kind that does not
 * apply may be null. */
qe_status qe_get_token(qe_handle h, int layer, int unit, int pos, int* tier, uint16_t* k_bf16, uint16_t* v_bf16,
                       uint8_t* k_codes, uint8_t* v_codes, float* params);

/* Number of kernel launches the handle has enqueued since qe_init. */
long long qe_kernel_launches(qe_handle h);

/* ---------------------------------------------------------------- fault injection (tests)
 *
 * Not part of the method on the pages (H2O page §5.1 asks for failure canaries and a fallback;
 * this is how the library's failure paths are exercised).  Every injection acts on the host or
 * on a wait whose data has already arrived: none faults, traps or hangs a GPU.
 *  QE_DEBUG_FAIL_DEVICE_ALLOC (h unused, may be NULL; process-wide): value n >= 1 makes the n-th
 *    device allocation of the next qe_init fail as out of memory: qe_init frees what it had
 *    allocated and returns QE_ERR_OOM naming the buffer.  0 clears.  One-shot.
 *  QE_DEBUG_FAIL_HOST_STORE (h unused; process-wide): value != 0 makes the pinned host backing
 *    store allocation of the next window-tiered qe_init fail: QE_ERR_HOST_STORE.  One-shot.
 *  QE_DEBUG_EXPIRE_WAIT (h required): value k >= 1: in the handle's next decode step
 *    (qe_decode_step of either tiering), every warp of the attention launch that streams at
 *    least k tiles reports its k-th tile wait as expired once that tile's copy has landed,
 *    lets its other copies land and leaves.  The sticky device flag then makes qe_synchronize
 *    return QE_ERR_TIMEOUT, as a real expiry (0.2 s without data) would; that step's outputs
 *    and score updates are undefined.  0 clears.
 *  QE_DEBUG_VERIFY_PATH (h required): which path qe_verify takes on the handle from now on:
 *    0 automatic (the default: the fused tensor-core launch when it is allowed and expected to
 *    be faster), 1 the fused launch whenever it is allowed (keys used as stored, n_q *
 *    group <= 64), 2 draft by draft.  Both paths compute the same results up to float32
 *    summation order; this lets tests cover each.  Not a fault: it persists until changed.
 * Errors: QE_ERR_INVALID_ARG (unknown kind, negative value, NULL handle for the wait or the
 * verify path, a path outside 0..2). */
enum { QE_DEBUG_FAIL_DEVICE_ALLOC = 1, QE_DEBUG_FAIL_HOST_STORE = 2, QE_DEBUG_EXPIRE_WAIT = 3,
       QE_DEBUG_VERIFY_PATH = 4 };
qe_status qe_debug_inject(qe_handle h, int what, long long value);

/* ---------------------------------------------------------------- snapshots (session restore)
 *
 * H2O page §6 (session restore): what a cache needs to resume is more than its K and V -- the
 * tiers, the cumulative scores (which the K and V cannot rebuild), the window boundaries,
 * positions and lengths.  A snapshot holds all of a window-tiered handle's state: the table
 * (tiers, slots, scores, lists, free stacks, victim and previous-slot marks), the bf16 and
 * 2-bit window slabs and their magnitude records, the pinned host store and ledger, the layer
 * headers, the routing counters and records, and each layer's host-side length and counts.
 * Split-K scratch, staging and verify deltas are rebuilt by every call and not saved.  The
 * format is this build's own (magic "QESNAP01"); it is not meant to cross builds or machines.
 *
 * qe_snapshot_size: bytes a snapshot of h takes (synchronous, no device work).
 * qe_snapshot: writes the snapshot into host (at least qe_snapshot_size bytes; any host
 *   memory).  Synchronous: a pending single-token append is written first, then the handle's
 *   stream is synchronised and the state copied out.
 * qe_restore: replaces h's whole state with a snapshot of a handle with the same
 *   configuration (every field that fixes the layout must match; QE_ERR_INVALID_ARG
 *   otherwise, h unchanged).  Synchronous; afterwards h continues exactly as the snapshotted
 *   handle would have: the same outputs, scores and tiers, bit for bit.
 * Errors: QE_ERR_STATE (a five-tier handle; a layer awaiting qe_verify_commit),
 * QE_ERR_INVALID_ARG (null pointers, a buffer too small, not a snapshot, another
 * configuration), QE_ERR_CUDA. */
qe_status qe_snapshot_size(qe_handle h, size_t* bytes);
qe_status qe_snapshot(qe_handle h, void* host, size_t bytes);
qe_status qe_restore(qe_handle h, const void* host, size_t bytes);

/* ---------------------------------------------------------------- no-allocation decode step
 *
 * Not part of the method on the pages (the paper has no counterpart): a library service.
 *
 * The same decode step as qe_decode_step (same kernels, same results up to the summation order
 * of the split-K merge), for callers that may not allocate device memory on the decode path:
 * callers whose device memory is owned by an arena or budget manager that forbids new
 * allocations once serving has started, callers for which a cudaMalloc could block on the
 * allocator or synchronise the device at the wrong moment, or threads that are not allowed to
 * make allocating CUDA calls.  It calls no cudaMalloc, cudaFree or other allocating routine:
 *  - q and out must be device memory ([batch][n_q_heads][head_dim] bf16 in, float32 or bf16
 *    out as configured); host pointers are not accepted (qe_decode_step would stage them
 *    through buffers it allocates on first use);
 *  - the split-K scratch comes from a fixed static device array inside the library (about
 *    4.1 MiB, held on every GPU that loads the library until the process exits), not from
 *    the handle.
 * Limits (QE_ERR_CAPACITY beyond them): batch * n_kv_heads <= 16 units; at most 8192 tiles per
 * unit (a tile is 16 bf16 tokens or one 2-bit window); G <= 4; head_dim <= 128.
 * The handle's device (the one current at qe_init) must be the current device at every call
 * (QE_ERR_STATE otherwise): the array's address is looked up, and used, for that device only.
 * The first call on each device looks up the array's device address (cudaGetSymbolAddress,
 * with that device current); make that first call before any stream capture.
 * QE_ERR_STATE too while the layer awaits qe_verify_commit, as for qe_decode_step.
 * qe_set_timing does not cover this entry point: its launches are not timed or counted by
 * qe_get_timing.  All calls share
 * the one array: calls whose work may overlap on the GPU (other streams, other handles on the
 * same device) race on it and must be serialised by the caller.  Nothing in the array needs to
 * start at zero: each call writes every scratch value it reads.  Like qe_decode_step, it counts
 * a pending single-token append, updates the window scores and is enqueued on the handle's
 * stream without waiting. */
qe_status qe_decode_step_noalloc(qe_handle h, int layer, const void* q, void* out);

#ifdef __cplusplus
}
#endif

#endif /* QE_H */
