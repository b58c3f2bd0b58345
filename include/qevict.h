/*
 * qevict.h — C ABI of the QEvict decode-time path on GB300 (sm_103a).
 *
 * QEvict ("QEvict: Recoverable Quantized KV Eviction for Attention-Drift-Robust
 * Long-Context Decoding", arXiv 2608.05326) keeps each layer's history as
 * contiguous windows in one of three tiers: Full (bf16), Quantized (INT2/INT4
 * codes with fp16 scale/offset, a write-once ledger) or Evicted, under a byte
 * budget.  Decoding attends over sink + Full + dequantised Quantized + recent
 * tokens, accumulates a per-window attention score, and every Omega generated
 * tokens re-ranks the windows and migrates them between tiers.
 *
 * Conventions for every entry point
 *   - Pointers named d_* / the arena / every tensor argument are DEVICE
 *     pointers unless stated otherwise; sizes are in bytes unless stated.
 *   - The caller owns all device memory: the arena, inputs and outputs.  The
 *     library never allocates device memory and keeps no pointer to inputs
 *     after a call returns.  The cache handle is host memory owned by the
 *     library (freed by qevict_destroy).
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default)
 *     and runs asynchronously; host-side argument checks are synchronous.
 *   - Errors: QEVICT_EINVAL for bad arguments, QEVICT_EBUDGET when the budget
 *     cannot hold the protected regions, QEVICT_ENOMEM for a too small arena,
 *     QEVICT_ESCHEDULE for a routing call off the Omega cadence, QEVICT_ECUDA
 *     when a launch fails, QEVICT_EDEVICE when a kernel recorded a fault in the
 *     device status word (read by qevict_read_counters / qevict_check).  On an
 *     error nothing is enqueued unless stated.  Bits of the status word: 1 a
 *     bounded wait ran out, 2 a routing event found too few free slots, 4 a
 *     kernel found the cache state inconsistent, 8 (checked build only,
 *     libqevict_check.so) an index read from device data was outside its buffer
 *     and its access was skipped; they stay set until an earlier export is
 *     imported or the cache is re-initialised.
 *   - Tensors are dense, row-major, bf16 (uint16 storage) unless stated.
 *   - One cache serves `batch` sequences that decode in lockstep and all
 *     `n_layers` layers; every (sequence, layer) pair is one independent "unit".
 */
#ifndef QEVICT_H
#define QEVICT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *qevict_stream_t; /* same type as cudaStream_t */

typedef enum {
  QEVICT_OK = 0,
  QEVICT_EINVAL = 1,
  QEVICT_EBUDGET = 2,
  QEVICT_ENOMEM = 3,
  QEVICT_ESCHEDULE = 4,
  QEVICT_ECUDA = 5,
  QEVICT_EDEVICE = 6
} qevict_status;

/* Sizes of one cache.  Semantics are per (sequence, layer); all units share them.
 * Supported: d_head = 128; (window, bits) in {(32, 2), (64, 4)}; h_q / h_kv in
 * {1, 2, 4, 8}; 1 <= n_sink <= 16; n_recent >= window; prompt_len > n_sink. */
typedef struct {
  int32_t batch, n_layers, h_q, h_kv, d_head;
  int32_t n_sink, n_recent, window, bits, omega;  /* omega: decode steps between routing events, 1..256 */
  int32_t q_num, q_den;           /* quantised-tier fraction q = q_num / q_den (QEvict §4.3 Eq. (3)) */
  int32_t budget_num, budget_den; /* B_total = floor(budget_num * M_FullKV / budget_den) when b_total == 0 */
  int64_t b_total;                /* bytes per (sequence, layer); 0 = use the fraction above */
  int32_t prompt_len, max_len;    /* max_len = prompt_len + decode steps the cache must hold */
  /* Window ranking at routing events (QEvict App. J; 0 everywhere = the paper's default):
   *   ranker 0: cumulative attention S += u per event (QEvict §4.2 Eq. (1), App. J Eq. (21));
   *   ranker 1: decayed attention S = decay * S + u (Eq. (22)); decay in (0, 1], 0 = 0.99;
   *   ranker 2: attention p-norm, ranked by sum over events of u^pnorm (Eq. (23)); pnorm >= 1, 0 = 3;
   *   ranker 3: key-vector norm, lower mean key L2 norm first (Eq. (24)), taken when the window
   *             leaves the recent region.
   * u is the window's attention since the previous event (App. J Eq. (20)).  no_promotion = 1:
   * quantized windows may be evicted but never return to the full tier (QEvict App. K). */
  int32_t ranker, no_promotion;
  float decay, pnorm;
  /* Key domain of the Quantized tier (QEvict §4.3, "Cache Execution"): 0 = keys are quantised as
   * given; 1 = the given keys carry rotate-half RoPE (pairs (i, i + 64), angle pos * theta_i) and
   * are quantised in the pre-RoPE domain, RoPE being re-applied at the window's positions after
   * dequantisation (attention and promotion).  rope = 1 needs qevict_set_rope_table before the
   * first prefill.  reserved0 must be 0. */
  int32_t rope, reserved0;
} qevict_config;

/* Byte budget of one (sequence, layer), QEvict §4.1 (constraint), §4.3 Eq. (3), App. B.4 Eq. (7)-(8).
 *   full_bytes = 2 * h_kv * d_head * prompt_len * 2           (bf16 K and V, Eq. (7) per layer)
 *   b_sink = n_sink * (c_tok + 4), b_local = (n_recent + window) * (c_tok + 4), c_tok = 4 * h_kv * d_head
 *   b_hist = b_total - b_sink - b_local
 *   payload = 2*h_kv*window*d_head*bits/8 + h_kv*d_head*4 + h_kv*window*4   (codes, fp16 scale/offset)
 *   m_q = payload + 4*window + 16;  m_f = window*c_tok + 4*window + 8 + payload (dormant-ledger reserve)
 *   k_f = floor((1-q) * b_hist / m_f),  k_q = floor(q * b_hist / m_q)      (exact integers)        */
typedef struct {
  int64_t full_bytes, b_total, b_sink, b_local, b_hist, payload, m_f, m_q;
  int32_t k_f, k_q;
  int32_t n_windows;      /* window ids 0 .. n_windows-1 can ever exist: ceil((max_len - n_sink) / window) */
  int32_t ring_windows;   /* windows of recent-region storage per unit */
} qevict_budget_info;

/* Where each part of the cache tuple lives inside the caller's arena, as byte
 * offsets from the arena base.  Unit u = layer * batch + seq; the region of unit u
 * starts at off_X + u * stride_X.  Layouts (all per unit):
 *   sink   [h_kv][2 (K,V)][n_sink][d_head] bf16, row-major                     (S of Eq. (2))
 *   ring   [h_kv][2][ring_windows][window*d_head] bf16 blocks, one block per
 *          window j at ring slot j % ring_windows, fragment-native (below)     (L_t)
 *   fpool  [k_f][h_kv][2][window*d_head] bf16 blocks, fragment-native          (F_t data)
 *   ledger [k_f+k_q][h_kv][qblock] bytes: K codes | V codes | K scale[d] | K offset[d] |
 *          V scale[window] | V offset[window] (fp16), qblock = payload / h_kv   (Q_t data, ledger Λ)
 *   score  [h_kv][n_windows] fp32: per-KV-head partial scores; the window score S(w) of
 *          QEvict §4.2 Eq. (1) is their sum over the KV heads (in head order), and right
 *          after a routing event the whole sum sits in head 0
 *   state  [n_windows] uint8: bits 0-1 tier (0 recent/unrouted, 1 Full, 2 Quantized, 3 Evicted),
 *          bits 2-3 ledger status (0 none, 1 active, 2 dormant)                  (E_t is tier 3)
 *   fslot, lslot [n_windows] int32: F-pool slot / ledger slot of a window, -1 if none
 *   ftab   [k_f] int32 pairs (window id, F slot), ascending window id; f_count valid
 *   qtab   [k_q] int32 pairs (window id, ledger slot), ascending window id; q_count valid
 *   meta   int32[16]: [0] tokens cached T, [1] windows routed so far, [2] f_count, [3] q_count
 *   agg    [n_windows] fp32: the ranker's value of every window for rankers 1-3 (the score
 *          region then holds only the attention since the last routing event)
 *
 * Fragment-native bf16 block of one window and KV head (W = window tokens, d = 128):
 *   K element (tok, dim), tok < W: index (((tok/16)*8 + dim/16)*32 + lane)*8 + reg*2 + (dim%2)
 *   V element (tok, dim):          index (((tok/16)*8 + dim/16)*32 + lane)*8 + reg*2 + (tok%2)
 *   where for K: r = tok%16, c = dim%16; for V: r = dim%16, c = tok%16;
 *   lane = (r%8)*4 + (c%8)/2 and reg = r/8 + 2*(c/8)  (the m16n8k16 A-operand register map).
 * Fragment-native INT2 codes (W = 32; 1 KB per K or V block): each of the 32 lanes owns 32 bytes,
 * stored as two 16-byte pieces at piece*512 + lane*16 + (byte%16), lane byte b -> piece b/16.
 *   K element (tok, dim): with r, c, lane, reg as above, group = (tok/16)*8 + dim/16,
 *     e = reg*2 + dim%2, bit = 4e (e < 4) or 4(e-4)+2 (e >= 4) inside the 16-bit field of
 *     (group, lane), which is lane bytes 2*group, 2*group+1 (little-endian).
 *   V element (tok, dim): with r = dim%16, c = tok%16 and lane as above, word i = dim/16 (lane
 *     bytes 4i .. 4i+3, little-endian), token pair tau = 2*(tok/16) + c/8,
 *     bit = 8*(r/8) + 2*tau + 16*(tok%2) inside that word.
 * Fragment-native INT4 codes (W = 64; 4 KB per K or V block): one little-endian 32-bit word per
 * (16x16 tile, lane), tile = (tok/16)*8 + dim/16, stored at word ((tile/4)*32 + lane)*4 + tile%4.
 *   K element (tok, dim): r = tok%16, c = dim%16, lane and reg as above, bits 4*(reg*2 + dim%2).
 *   V element (tok, dim): r = dim%16, c = tok%16, lane and reg as above, bits 4*reg + 16*(tok%2).
 * A W = 64 ledger record (qblock 8960 B) is K codes | V codes | parameters, each code block 4 KB.
 */
typedef struct {
  int64_t off_sink, stride_sink;
  int64_t off_ring, stride_ring;
  int64_t off_fpool, stride_fpool;
  int64_t off_ledger, stride_ledger;
  int64_t off_score, stride_score;
  int64_t off_state, stride_state;
  int64_t off_fslot, stride_fslot;
  int64_t off_lslot, stride_lslot;
  int64_t off_ftab, stride_ftab;
  int64_t off_qtab, stride_qtab;
  int64_t off_meta, stride_meta;
  int64_t qblock;        /* ledger bytes per (slot, KV head) */
  int64_t arena_bytes;
  int32_t n_split;       /* decode split-K partitions per (sequence, KV head) */
  int32_t pad_;
  int64_t off_agg, stride_agg;
  int64_t off_rope;      /* rope = 1: fp32 [max_len][64][2] (cos, sin) table shared by all units */
} qevict_layout;

typedef struct qevict_cache qevict_cache;

/* Validates cfg and fills the budget of one (sequence, layer).  Host only. */
qevict_status qevict_budget(const qevict_config *cfg, qevict_budget_info *out);

/* Bytes of device arena a cache of this configuration needs (256-byte aligned base required). */
qevict_status qevict_cache_bytes(const qevict_config *cfg, size_t *bytes);

/* Creates a cache over the caller's arena (d_arena, at least qevict_cache_bytes bytes, 256-byte
 * aligned) and enqueues its zero/-1 initialisation on `stream`.  *out receives a host handle. */
qevict_status qevict_init_cache(const qevict_config *cfg, void *d_arena, size_t bytes,
                                qevict_stream_t stream, qevict_cache **out);

/* Region offsets of the cache tuple inside the arena (see qevict_layout).  Host only. */
qevict_status qevict_get_layout(const qevict_cache *cache, qevict_layout *out);

/* RoPE table of a rope = 1 cache (QEvict §4.3: quantised keys keep their absolute positions and
 * are rotated again after dequantisation).  d_table: fp32 [rows][64][2] on the device, row p
 * holding (cos(p * theta_i), sin(p * theta_i)) for i = 0..63, the angles the caller's model used to
 * rotate its keys; rows >= max_len.  The first max_len rows are copied into the arena on `stream`
 * (the caller keeps ownership of d_table).  Keys are taken back with
 *   x_i c + x_{i+64} s,  x_{i+64} c - x_i s    and rotated with    x_i c - x_{i+64} s,  x_{i+64} c + x_i s,
 * every product and sum rounded to fp32 on its own.  QEVICT_EINVAL when the cache has rope = 0 or
 * rows < max_len; call before the first qevict_prefill_route (later calls return QEVICT_ESCHEDULE). */
qevict_status qevict_set_rope_table(qevict_cache *cache, const float *d_table, int64_t rows, qevict_stream_t stream);

/* Prompt scoring, QEvict §4.2 (last paragraph): for every (sequence, window j starting in the
 * prompt) S0[j] = (1/h_q) sum_h sum_{tau < P} sum_{i in w_j, i <= tau} a_tau^h(i), dense causal
 * attention of every prompt query.  q_prompt [batch][P][h_q][d], k_prompt [batch][P][h_kv][d];
 * s0_out [batch][ceil((P - n_sink) / window)] fp32.  Prompts are per layer: call once per layer.
 * q_prompt and k_prompt must be 16-byte aligned (TMA tensor maps), else QEVICT_EINVAL.
 * Scratch: a region of the arena reserved for it (no allocation); reads the inputs twice. */
qevict_status qevict_prefill_scores(const qevict_cache *cache, const void *q_prompt, const void *k_prompt,
                                    float *s0_out, qevict_stream_t stream);

/* Prefill of one layer, QEvict §4.2 (last paragraph) and §4.3 Eq. (2)-(5): stores the sink and the
 * recent region, sets the window scores (s0 [batch][ceil((P - n_sink)/window)] fp32, or computed
 * from q_prompt when s0 is NULL), routes all historical prompt windows into F / Q / E and
 * materialises F (bf16 copy) and Q (quantised once).  k_prompt, v_prompt [batch][P][h_kv][d].
 * Must be called exactly once per layer, before any decode step of that layer.  A rope = 1 cache
 * needs its RoPE table first (QEVICT_ESCHEDULE otherwise).  k_prompt and v_prompt must be 2-byte,
 * s0 4-byte and (when s0 is NULL) q_prompt and k_prompt 16-byte aligned, else QEVICT_EINVAL. */
qevict_status qevict_prefill_route(qevict_cache *cache, int32_t layer, const void *k_prompt,
                                   const void *v_prompt, const float *s0, const void *q_prompt,
                                   qevict_stream_t stream);

/* One decode step of one layer for every sequence, QEvict §4.1 (attention over the accessible
 * set) and §4.2 Eq. (1): appends k_new, v_new [batch][h_kv][d] at position T (the recent region),
 * computes out[batch][h_q][d] = softmax(q K_acc^T / sqrt(d)) V_acc over sink + Full + dequantised
 * Quantized + recent tokens (the new token included; query head h reads KV head h / (h_q/h_kv)),
 * and records the attention mass of every accessible non-sink window.  The window scores absorb
 * these masses, (1/h_q) * sum_h (mass of window w) per step and in step order, at the next
 * qevict_flush_scores or qevict_route.  q [batch][h_q][d].  Fails with QEVICT_ESCHEDULE if the
 * cache is full (T = max_len) or a routing event is due, with QEVICT_EINVAL if q or k_new is not
 * 4-byte aligned or v_new or out is not 2-byte aligned. */
qevict_status qevict_decode_step(qevict_cache *cache, int32_t layer, const void *q, const void *k_new,
                                 const void *v_new, void *out, qevict_stream_t stream);

/* Routing event for every layer and sequence, QEvict §4.3 Eq. (4)-(6) and App. A Algorithm 1:
 * candidates = Full + Quantized + windows aged out of the recent region; rank by score
 * (descending, ties to the older window); first k_f -> Full, next k_q -> Quantized, rest ->
 * Evicted.  Quantises newly demoted windows once (reusing a dormant ledger when one exists),
 * rebuilds promoted windows in bf16 from their ledger, copies aged windows, frees evicted ones,
 * and rebuilds the F / Q tables in window order with the lowest free slots going to new windows
 * in window order.  Legal only when every layer has taken the same multiple of omega decode
 * steps since its prefill (else QEVICT_ESCHEDULE). */
qevict_status qevict_route(qevict_cache *cache, qevict_stream_t stream);

/* QEvict §4.2 Eq. (1), applied lazily: adds the window masses recorded by every decode step since
 * the previous flush (of any layer) to the window scores, one step at a time in decode order, so
 * the scores equal those of an update after every step.  qevict_route flushes by itself; call this
 * only to read scores between routing events.  QEVICT_ESCHEDULE before every layer is prefilled. */
qevict_status qevict_flush_scores(qevict_cache *cache, qevict_stream_t stream);

/* Copies the 7 cumulative transition counters (promotions Q->F, demotions F->Q, first-time
 * quantisations, ledger reactivations, evictions, aged->F, aged->Q), summed over all units, to
 * host memory `host7`.  Synchronises `stream`.  Returns QEVICT_EDEVICE if a kernel recorded a
 * fault in the device status word. */
qevict_status qevict_read_counters(qevict_cache *cache, int64_t *host7, qevict_stream_t stream);

/* Synchronises `stream`, re-reads the per-layer token counts (needed after replaying captured
 * CUDA graphs of decode steps) and returns QEVICT_EDEVICE if the device status word is set. */
qevict_status qevict_check(qevict_cache *cache, qevict_stream_t stream);

/* The device status word itself (its bits are listed with the conventions above), copied to
 * *host_word after `stream` synchronises; the word is not cleared.  QEVICT_ECUDA if the copy fails. */
qevict_status qevict_read_status(const qevict_cache *cache, int32_t *host_word, qevict_stream_t stream);

/* Failure-reporting self-test.  Enqueues on `stream` a one-thread kernel that waits, through the
 * same bounded wait every kernel of the library uses, on an mbarrier phase that nothing completes.
 * After the wait's limit (about 200 ms) the kernel records a timeout in the cache's device status
 * word and returns; no GPU fault is raised and the context stays usable.  Nothing else in the cache
 * changes.  The next qevict_check / qevict_read_counters returns QEVICT_EDEVICE; the word stays set
 * until an exported state taken before it is imported (the status word travels in the arena) or the
 * cache is re-initialised.  Returns QEVICT_ECUDA if the launch fails. */
qevict_status qevict_selftest_wait(qevict_cache *cache, qevict_stream_t stream);

/* Test hook for the router's slot-exhaustion guard (QEvict App. A Algorithm 1, slot allocation of
 * newcomers to F and to the ledger).  With cap >= 0, every later routing event sees at most `cap`
 * free F slots and at most `cap` free ledger slots; cap = -1 (the default) removes the limit.  Real
 * pools cannot run out (a newcomer to F or Q always finds a slot released for it), so the guard is
 * reachable only this way.  An event whose newcomers need more slots than it sees sets bit 2 of
 * the device status word (qevict_check then returns QEVICT_EDEVICE) and changes no tier, slot,
 * table or ledger; its pending window masses are still absorbed into the scores.  Host only: nothing is enqueued.  QEVICT_EINVAL if cap < -1. */
qevict_status qevict_debug_cap_free_slots(qevict_cache *cache, int32_t cap);

/* Scratch size, in floats, of qevict_prefill_scores_noalloc: 2 * batch * h_q * prompt_len must not
 * exceed it (2 Mi floats = 8 MiB, e.g. 32 query heads x 32768 prompt tokens for one sequence). */
#define QEVICT_NOALLOC_SCRATCH_FLOATS (2LL * 1024 * 1024)

/* Prefill scores without any device allocation (the paper has no counterpart; this is an
 * interface for callers).  Computes exactly what qevict_prefill_scores computes, but takes plain
 * sizes instead of a cache, for callers that cannot allocate device memory at all: code inside a
 * framework that owns every byte of device memory through its own pool, or plugins handed only their
 * input and output buffers.  Its scratch is a fixed 8 MiB array inside the library image, held on
 * every GPU that loads the library until the process exits; nothing is allocated per call.
 *   q_prompt [batch][prompt_len][h_q][128], k_prompt [batch][prompt_len][h_kv][128] bf16 (device);
 *   s0_out [batch][ceil((prompt_len - n_sink) / window)] fp32 (device).  q_prompt, k_prompt 16-byte
 *   aligned, s0_out 4-byte aligned.
 * Errors: QEVICT_EINVAL for bad sizes, NULL or misaligned pointers; QEVICT_ENOMEM when
 * 2 * batch * h_q * prompt_len > QEVICT_NOALLOC_SCRATCH_FLOATS (nothing is enqueued then).
 * Device failures (a bounded wait of the scoring kernels that ran out) are not returned by this
 * asynchronous call: they set a device status word of this entry point, which
 * qevict_prefill_scores_noalloc_status reads and clears.
 * The first call on a device looks up the scratch address with that device current; make that first
 * call before capturing a stream.  All calls share the scratch: calls that can overlap on the GPU
 * (e.g. on two streams) race and must be ordered by the caller. */
qevict_status qevict_prefill_scores_noalloc(int32_t batch, int32_t prompt_len, int32_t h_q, int32_t h_kv,
                                            int32_t n_sink, int32_t window, const void *q_prompt,
                                            const void *k_prompt, float *s0_out, qevict_stream_t stream);

/* The device status word of qevict_prefill_scores_noalloc on the current device: synchronises
 * `stream`, reads the word and clears it (a device-to-host copy and a memset of the word; nothing is
 * allocated).  Returns QEVICT_EDEVICE if any call since the last read recorded a device failure,
 * whose s0_out must then be discarded; QEVICT_OK otherwise; QEVICT_ECUDA if the copy fails.  The
 * word is sticky until read: a failure of an earlier call is reported even after later calls. */
qevict_status qevict_prefill_scores_noalloc_status(qevict_stream_t stream);

/* Device views of one unit's cache tuple, QEvict §4.1 Eq. (2): C_t = (S, L_t, F_t, Q_t, E_t) of
 * (layer, seq).  Each pointer is the unit's region inside the arena, with the layout documented
 * with the layout struct above; E_t is the set of windows whose state tier is 3.  Host only;
 * nothing is enqueued. */
typedef struct {
  void *sink;        /* S:   [h_kv][2][n_sink][d] bf16 */
  void *ring;        /* L_t: recent windows, fragment-native bf16 blocks */
  void *fpool;       /* F_t data: [k_f][h_kv][2][window*d] fragment-native bf16 */
  void *ledger;      /* Q_t data and dormant ledgers: [k_f+k_q][h_kv][qblock] */
  float *score;      /* [h_kv][n_windows] per-KV-head partial scores */
  uint8_t *state;    /* [n_windows] tier (bits 0-1) and ledger status (bits 2-3) */
  int32_t *f_slot;   /* [n_windows] F-pool slot or -1 */
  int32_t *l_slot;   /* [n_windows] ledger slot or -1 */
  int32_t *f_table;  /* [k_f] (window id, F slot), ascending window id; meta[2] entries valid */
  int32_t *q_table;  /* [k_q] (window id, ledger slot), ascending window id; meta[3] entries valid */
  int32_t *meta;     /* [16]: [0] T, [1] windows routed, [2] f_count, [3] q_count, [6] routing events,
                        [7] T when the scores last absorbed the decode steps' masses */
} qevict_tuple;
qevict_status qevict_get_tuple(const qevict_cache *cache, int32_t layer, int32_t seq, qevict_tuple *out);

/* Checkpoint / resume (the paper has none; an interface for serving systems).  The export is a
 * header (format tag, the cache configuration, the arena size) followed by a byte copy of the whole
 * arena, pending decode-step mass records and counters included, written to HOST memory.
 * qevict_export_bytes gives its size.  qevict_export_state synchronises `stream` after the copy
 * (QEVICT_ENOMEM when `bytes` is too small).  qevict_import_state loads an export into a cache
 * created with the identical configuration (else QEVICT_EINVAL), synchronises `stream`, and resumes
 * its host bookkeeping (per-layer T, routing events) from the imported meta records.  A rope = 1
 * cache's RoPE table is part of the arena; an export taken before any prefill needs
 * qevict_set_rope_table again after its import. */
qevict_status qevict_export_bytes(const qevict_cache *cache, size_t *bytes);
qevict_status qevict_export_state(const qevict_cache *cache, void *host_buf, size_t bytes, qevict_stream_t stream);
qevict_status qevict_import_state(qevict_cache *cache, const void *host_buf, size_t bytes, qevict_stream_t stream);

/* Routing diagnostics against a FullKV run, QEvict App. I and App. K.  Two caches decode the same
 * inputs: `policy`, the cache evaluated (cumulative ranker, ranker = 0), and `fullkv`, a cache of the
 * same shapes whose budget keeps every window Full (its k_f >= n_windows), so its per-step window
 * masses are the FullKV attention A_tau(w).  Windows play the role of the pages' token positions.
 * At every routing event the diagnostics record, per (layer, sequence):
 *   FMM_H   App. I.2 Eq. (13): over the next `horizon` decode steps, the FullKV attention of each query
 *           head on the windows the policy holds Evicted, over that on every state that existed at
 *           the event (sinks and windows whose first position was cached); averaged over the
 *           (head, event) pairs whose horizon was fully decoded;
 *   churn   Eq. (14): Jaccard distance of the windows retained (Full or Quantized) at consecutive
 *           events;
 *   mu(z)   Eq. (15): shares of the FullKV window scores per policy tier (Full, Quantized, Evicted,
 *           Local) over the windows that exist, at the last event;
 *   QSA, R_Q  Eq. (16)-(17): cosine and sum ratio of the policy's and the FullKV window scores over
 *           the policy's Quantized windows, at events after the prefill;
 *   Global LIR(m)  Eq. (18): inactive episodes (runs of events outside the selected set that start
 *           when a window leaves it) that reach m events, and those that later return; for the
 *           policy's Full tier and for the FullKV top-k_f selection (ties to the older window);
 *   P_ab(Delta)  Eq. (19): counts of event pairs Delta = 1..8 apart with the window in (1) or out
 *           (0) of the policy's Full tier, counted from the event the window was first routed.
 * The diagnostics own no device memory: `d_buf` (256-byte aligned, qevict_diag_bytes long) holds
 * their state.  Errors: QEVICT_EINVAL for mismatched caches, a policy ranker other than 0, a FullKV
 * cache that can evict, horizon not a multiple of omega or above 8 * omega, lir_m < 0;
 * QEVICT_ESCHEDULE unless both caches are prefilled with no decode step yet (init) or both are due
 * for a routing event (qevict_diag_route). */
typedef struct qevict_diag qevict_diag;
typedef struct {
  int32_t horizon;   /* FMM horizon H in decode steps; 0 = 32 */
  int32_t lir_m;     /* Global LIR eligibility threshold m; 0 = 3 */
} qevict_diag_config;
typedef struct {
  int64_t events;                /* routing events recorded, the prefill's included */
  double fmm;                    /* mean FMM_H over its terms */
  int64_t fmm_terms;             /* (layer, sequence, query head, event) terms with a complete horizon */
  double churn;                  /* mean over consecutive event pairs of every unit */
  int64_t churn_terms;
  double qsa, r_q;               /* means over the events after the prefill with Quantized windows */
  int64_t qsa_terms;
  double tier_mass[4];           /* Full, Quantized, Evicted, Local shares at the last event, mean over units */
  int64_t lir_eligible, lir_rescued;                 /* policy Full tier */
  int64_t lir_fullkv_eligible, lir_fullkv_rescued;   /* FullKV top-k_f selection */
  int64_t lag[8][2][2];          /* lag[Delta-1][a][b] */
} qevict_diag_report;
qevict_status qevict_diag_bytes(const qevict_cache *policy, const qevict_diag_config *dc, size_t *bytes);
/* Records the prefill routing as the first event (enqueued on `stream`). */
qevict_status qevict_diag_init(qevict_cache *policy, qevict_cache *fullkv, const qevict_diag_config *dc, void *d_buf,
                               size_t bytes, qevict_stream_t stream, qevict_diag **out);
/* A routing event of both caches in place of two qevict_route calls: reads the FullKV masses of the
 * steps since the previous event, routes the policy, routes the FullKV cache, records the event.
 * The schedule of both caches is checked before anything is enqueued (QEVICT_ESCHEDULE); a launch
 * failure after that (QEVICT_ECUDA) leaves the caches and the diagnostics out of step. */
qevict_status qevict_diag_route(qevict_diag *diag, qevict_stream_t stream);
/* Synchronises `stream` and sums the per-unit records into `out` (host memory). */
qevict_status qevict_diag_read(qevict_diag *diag, qevict_diag_report *out, qevict_stream_t stream);
qevict_status qevict_diag_destroy(qevict_diag *diag);

/* Frees the host handle (the arena stays the caller's). */
qevict_status qevict_destroy(qevict_cache *cache);

const char *qevict_status_string(qevict_status status);

#ifdef __cplusplus
}
#endif

#endif /* QEVICT_H */
