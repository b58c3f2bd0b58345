"""CPU oracle for QEvict's decode-time path.  TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may import
this module.  The product path (the CUDA library and its Python binding) never
calls it, and it shares no code, table or constant generator with the CUDA
sources.

What it computes, each step cited to "QEvict: Recoverable Quantized KV Eviction
for Attention-Drift-Robust Long-Context Decoding" (arXiv 2608.05326, abbreviated
"QEvict") or to the review of the same paper on liuzhao09.github.io
("QEvict review"):

  * accessible-set GQA attention and per-window attention mass
        QEvict §4.1 (unnumbered attention equation), §4.2 Eq. (1)
  * window partition, tier state, byte-budget capacities
        QEvict §4.1, §4.3 Eq. (2), Eq. (3); App. B.4 Eq. (7), Eq. (8)
  * KIVI-style asymmetric low-bit quantisation, write-once ledger
        QEvict §4.3 "Migration-Stable Quantization"
  * candidate pool, TopK routing, state machine, migration
        QEvict §4.3 Eq. (4), Eq. (5), Eq. (6); App. A Algorithm 1
  * prefill scoring (prompt attention initialises the scores)
        QEvict §4.2 last paragraph

Arithmetic: attention, probabilities and masses in float64; the quantiser in
float32 with IEEE division and round-half-to-even, scale and offset stored as
float16; dequantised values rounded to bf16 (the model's execution datatype,
QEvict §4.3).  Readings taken where the pages are silent are stated beside the
code that takes them.

Parity pins (independent checks of this oracle) live in tests/test_oracle_*.py.
Parity unpinned: the paper's quality numbers and its diagnostic K_f/K_q values
for the R3/R4 policies (QEvict App. I.1), which need model traces.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional, Tuple

import numpy as np

# tier states of a routed window (QEvict §4.1: z(w) in {Full, Quantized, Evicted});
# LOCAL marks a window whose tokens are still in the protected recent region.
LOCAL, FULL, QUANT, EVICTED = 0, 1, 2, 3
# ledger status (QEvict App. A Algorithm 1: create, mark dormant, reactivate, delete)
NO_LEDGER, ACTIVE, DORMANT = 0, 1, 2

COUNTER_NAMES = ("promotions", "demotions", "first_quant", "reactivations", "evictions", "aged_full", "aged_quant")


# --------------------------------------------------------------------------- number formats

def bf16_round(x) -> np.ndarray:
    """Round float32 values to the nearest bf16 value, ties to even; returned as float32.

    bf16 keeps the upper 16 bits of the IEEE binary32 pattern; rounding adds
    0x7FFF plus the lowest kept bit before truncating (the usual RNE bit rule).
    """
    x = np.asarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    keep = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + keep) >> np.uint64(16)) << np.uint64(16)
    out = (r & np.uint64(0xFFFFFFFF)).astype(np.uint32).view(np.float32)
    return np.where(np.isnan(x), x, out).astype(np.float32)


def fp16_round(x) -> np.ndarray:
    """Round float32 values to IEEE binary16 (round-to-nearest-even)."""
    return np.asarray(x, dtype=np.float32).astype(np.float16)


# --------------------------------------------------------------------------- configuration

@dataclasses.dataclass(frozen=True)
class Config:
    h_q: int
    h_kv: int
    d_head: int = 128
    n_sink: int = 4
    n_recent: int = 128
    window: int = 32
    bits: int = 2
    omega: int = 8
    q_num: int = 70
    q_den: int = 100
    budget_num: int = 20
    budget_den: int = 100
    prompt_len: int = 4096
    max_len: int = 4160
    b_total: Optional[int] = None    # bytes per (sequence, layer); None = budget fraction of full KV
    # window ranking (QEvict App. J): 0 cumulative attention (the default, Eq. (21)), 1 exponentially
    # decayed attention (Eq. (22)), 2 attention p-norm (Eq. (23)), 3 key-vector norm (Eq. (24))
    ranker: int = 0
    decay: float = 0.99
    pnorm: float = 3.0
    # QEvict App. K: 1 = quantized windows may be evicted but never return to the full tier
    no_promotion: int = 0
    # QEvict §4.3: > 0 keeps quantized keys in the pre-RoPE domain (rotate-half RoPE, this base)
    # and re-rotates them at their positions after dequantisation; 0 = keys carry no rotation
    rope_base: float = 0.0

    @staticmethod
    def from_obj(o, **kw) -> "Config":
        fields = {f.name for f in dataclasses.fields(Config)}
        vals = {k: getattr(o, k) for k in fields if hasattr(o, k)}
        if "max_len" not in vals and hasattr(o, "steps"):
            vals["max_len"] = o.prompt_len + o.steps
        vals.update(kw)
        return Config(**vals)

    @property
    def group(self) -> int:
        return self.h_q // self.h_kv

    def n_windows_cap(self) -> int:
        return max(1, -(-(self.max_len - self.n_sink) // self.window))


# --------------------------------------------------------------------------- budget

@dataclasses.dataclass(frozen=True)
class Budget:
    full_bytes: int     # M_FullKV of one (sequence, layer) at the prompt length
    b_total: int
    b_sink: int
    b_local: int
    b_hist: int
    payload: int        # quantised bytes of one window: codes + scales/offsets
    m_f: int
    m_q: int
    k_f: int
    k_q: int


def budget(cfg: Config) -> Budget:
    """Byte budget and tier capacities of one (sequence, layer).

    M_FullKV = 2 * H_kv * d_h * S * c_f per layer with c_f = 2 bytes
    (QEvict App. B.4 Eq. (7), taken per layer and per sequence, S = prompt length).
    B_total = floor(fraction * M_FullKV) unless given in bytes.
    Protected regions (QEvict §4.1): the sink tokens and a recent region charged
    at n_recent + W tokens (the largest local region left after a routing event),
    each token at its bf16 K and V plus an int32 position (App. B.4 Eq. (8), M_position).
    Per-window costs (QEvict §4.3 "Byte-Constrained Tier Allocation": packed codes,
    quantisation parameters, positions and persistent indexing state):
      M_q = payload + W positions * 4 + 16 bytes of ledger/table record,
      payload = 2*H_kv*W*d*BITS/8 code bytes + H_kv*d*(2+2) key scale/offset (fp16,
                per channel) + H_kv*W*(2+2) value scale/offset (fp16, per token);
      M_f = W * bf16 K+V + W positions * 4 + 8 bytes of table record + payload.
    The payload inside M_f reserves the dormant ledger a promoted window keeps
    (Algorithm 1 marks it dormant instead of deleting it), so the budget holds
    for every mix of tiers.
    Capacities, QEvict §4.3 Eq. (3), with q = q_num / q_den in exact integers:
      K_f = floor((1 - q) * B_hist / M_f),  K_q = floor(q * B_hist / M_q).
    """
    c_tok = 2 * cfg.h_kv * cfg.d_head * 2
    tok_bytes = c_tok + 4
    full = c_tok * cfg.prompt_len
    b_total = cfg.b_total if cfg.b_total is not None else full * cfg.budget_num // cfg.budget_den
    b_sink = cfg.n_sink * tok_bytes
    b_local = (cfg.n_recent + cfg.window) * tok_bytes
    b_hist = b_total - b_sink - b_local
    if b_hist < 0:
        raise ValueError("budget below the protected sink and recent bytes")
    payload = (2 * cfg.h_kv * cfg.window * cfg.d_head * cfg.bits // 8
               + cfg.h_kv * cfg.d_head * 4 + cfg.h_kv * cfg.window * 4)
    m_q = payload + cfg.window * 4 + 16
    m_f = cfg.window * c_tok + cfg.window * 4 + 8 + payload
    k_f = (cfg.q_den - cfg.q_num) * b_hist // (cfg.q_den * m_f)
    k_q = cfg.q_num * b_hist // (cfg.q_den * m_q)
    return Budget(full, b_total, b_sink, b_local, b_hist, payload, m_f, m_q, k_f, k_q)


def n_hist(T: int, cfg: Config) -> int:
    """Windows that have left the recent region when T tokens are cached.

    Windows are W contiguous tokens aligned at the end of the sink prefix
    (QEvict §4.1: the history after the sink and recent regions is split into
    contiguous windows).  Reading: window j = [n_s + jW, n_s + (j+1)W) has aged
    once its last token is at least n_recent tokens old.
    """
    return max(0, (T - cfg.n_recent - cfg.n_sink) // cfg.window)


def prompt_windows(cfg: Config) -> int:
    """Windows that start inside the prompt (the last one may be partial)."""
    return max(0, -(-(cfg.prompt_len - cfg.n_sink) // cfg.window))


def window_of(pos: int, cfg: Config) -> int:
    return -1 if pos < cfg.n_sink else (pos - cfg.n_sink) // cfg.window


# --------------------------------------------------------------------------- quantisation

def quantize_groups(x: np.ndarray, axis: int, bits: int):
    """Asymmetric min/max quantisation of bf16 values along `axis`.

    One group per slice along `axis` (QEvict §4.3: keys per channel across the
    tokens, values per token across the channels).  Reading of the rounding:
      mn, mx       exact float32 of the group's bf16 extremes
      s32          (mx - mn) / (2^BITS - 1)        float32, IEEE division
      s, m         float16(s32), float16(mn)       stored parameters
      code         clamp(rint((x - m) / s), 0, 2^BITS - 1), float32 arithmetic,
                   ties to even; code = 0 where s == 0 (constant group)
    Returns integer codes shaped like x and float16 s, m with `axis` removed.
    """
    x = np.asarray(x, dtype=np.float32)
    levels = np.float32((1 << bits) - 1)
    mn = x.min(axis=axis)
    mx = x.max(axis=axis)
    s32 = (mx - mn) / levels
    s16 = fp16_round(s32)
    m16 = fp16_round(mn)
    s = np.expand_dims(s16.astype(np.float32), axis)
    m = np.expand_dims(m16.astype(np.float32), axis)
    with np.errstate(divide="ignore", invalid="ignore"):
        t = (x - m) / s
    code = np.clip(np.rint(t), np.float32(0), levels)
    code = np.where(s == 0, np.float32(0), code)
    return code.astype(np.uint8), s16, m16


def dequantize_groups(code: np.ndarray, s16: np.ndarray, m16: np.ndarray, axis: int) -> np.ndarray:
    """x_hat = bf16(float32(code * s + m)): the same low-bit approximation rebuilt in the
    execution datatype (QEvict §4.3: promotion reconstructs it in the model's datatype).
    code * s is exact in float32 (code < 16, s has 11 significant bits), so the float32
    sum is rounded once, as a fused multiply-add would round it."""
    s = np.expand_dims(np.asarray(s16).astype(np.float32), axis)
    m = np.expand_dims(np.asarray(m16).astype(np.float32), axis)
    return bf16_round(code.astype(np.float32) * s + m)


def rope_rotate(x: np.ndarray, cs: np.ndarray, inverse: bool = False) -> np.ndarray:
    """Rotate-half RoPE of d = 128 vectors (QEvict §4.3 re-applies RoPE after dequantisation).

    x [..., 128]; cs [..., 64, 2] holds (cos, sin) of pos * theta_i for the pairs (i, i + 64),
    broadcast against x's leading axes.  Forward: x_i c - x_{i+64} s and x_{i+64} c + x_i s;
    inverse (back to the pre-RoPE domain): x_i c + x_{i+64} s and x_{i+64} c - x_i s.  Float32,
    every product and every sum rounded on its own (no fused multiply-add)."""
    x = np.asarray(x, np.float32)
    a, b = x[..., :64], x[..., 64:]
    c, sn = np.asarray(cs[..., 0], np.float32), np.asarray(cs[..., 1], np.float32)
    if inverse:
        return np.concatenate([a * c + b * sn, b * c - a * sn], axis=-1).astype(np.float32)
    return np.concatenate([a * c - b * sn, b * c + a * sn], axis=-1).astype(np.float32)


@dataclasses.dataclass
class Ledger:
    """Write-once quantised record of one window (QEvict §4.3, Algorithm 1 Λ_w).

    Arrays are per KV head: codes_k/codes_v [H_kv][W][d]; key parameters per
    channel [H_kv][d]; value parameters per token [H_kv][W]."""
    codes_k: np.ndarray
    s_k: np.ndarray
    m_k: np.ndarray
    codes_v: np.ndarray
    s_v: np.ndarray
    m_v: np.ndarray
    status: int = ACTIVE
    slot: int = -1

    def dequantize(self, cs: Optional[np.ndarray] = None) -> Tuple[np.ndarray, np.ndarray]:
        """Returns K_hat, V_hat as [W][H_kv][d] float32 (bf16 values).  With cs ([W][64][2], the
        window's positions) the pre-RoPE keys are re-rotated and rounded to bf16 (QEvict §4.3)."""
        k = dequantize_groups(self.codes_k, self.s_k, self.m_k, axis=1)   # [H][W][d]
        v = dequantize_groups(self.codes_v, self.s_v, self.m_v, axis=2)
        k = k.transpose(1, 0, 2).copy()
        if cs is not None:
            k = bf16_round(rope_rotate(k, np.asarray(cs)[:, None, :, :]))
        return k, v.transpose(1, 0, 2).copy()


def quantize_window(K: np.ndarray, V: np.ndarray, bits: int, cs: Optional[np.ndarray] = None) -> Ledger:
    """K, V: [W][H_kv][d] bf16 values as float32.  With cs ([W][64][2]) the keys, which carry their
    positions' rotation, are first taken back to the pre-RoPE domain and quantised there."""
    if cs is not None:
        K = rope_rotate(K, np.asarray(cs)[:, None, :, :], inverse=True)
    kh = np.asarray(K, np.float32).transpose(1, 0, 2)   # [H][W][d]
    vh = np.asarray(V, np.float32).transpose(1, 0, 2)
    ck, sk, mk = quantize_groups(kh, axis=1, bits=bits)   # per (head, channel) over tokens
    cv, sv, mv = quantize_groups(vh, axis=2, bits=bits)   # per (head, token) over channels
    return Ledger(ck, sk, mk, cv, sv, mv)


# --------------------------------------------------------------------------- attention

def attend(q: np.ndarray, K: np.ndarray, V: np.ndarray, h_kv: int):
    """a^h = softmax(q^h K^T / sqrt(d)), o^h = a^h V over the given tokens (QEvict §4.1).

    q [H_q][d]; K, V [N][H_kv][d].  GQA reading: query head h reads KV head
    floor(h / (H_q / H_kv)).  Returns o [H_q][d] and a [H_q][N], both float64.
    """
    q = np.asarray(q, np.float64)
    K = np.asarray(K, np.float64)
    V = np.asarray(V, np.float64)
    h_q, d = q.shape
    G = h_q // h_kv
    o = np.zeros((h_q, d))
    a = np.zeros((h_q, K.shape[0]))
    for h in range(h_q):
        g = h // G
        logits = K[:, g, :] @ q[h] / np.sqrt(d)
        e = np.exp(logits - logits.max())
        a[h] = e / e.sum()
        o[h] = a[h] @ V[:, g, :]
    return o, a


def prefill_scores(q: np.ndarray, k: np.ndarray, cfg: Config, row_block: int = 512) -> np.ndarray:
    """Initial window scores from prompt attention (QEvict §4.2, last paragraph).

    Reading: every prompt query attends causally (token tau sees i <= tau);
    S_0[j] = (1/H_q) * sum_h sum_tau sum_{i in w_j, i <= tau} a_tau^h(i), for every
    window j that starts inside the prompt (partial windows included, sinks excluded).
    q [P][H_q][d], k [P][H_kv][d].
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    P, h_q, d = q.shape
    G = h_q // cfg.h_kv
    col = np.zeros(P)
    for h in range(h_q):
        kg = k[:, h // G, :]
        for r0 in range(0, P, row_block):
            r1 = min(P, r0 + row_block)
            logits = q[r0:r1, h, :] @ kg[:r1].T / np.sqrt(d)        # [rows][r1]
            mask = np.arange(r1)[None, :] > np.arange(r0, r1)[:, None]
            logits[mask] = -np.inf
            e = np.exp(logits - logits.max(axis=1, keepdims=True))
            a = e / e.sum(axis=1, keepdims=True)
            col[:r1] += a.sum(axis=0)
    n_win = -(-(P - cfg.n_sink) // cfg.window) if P > cfg.n_sink else 0
    S0 = np.zeros(n_win)
    for j in range(n_win):
        lo = cfg.n_sink + j * cfg.window
        S0[j] = col[lo:min(P, lo + cfg.window)].sum() / h_q
    return S0


# --------------------------------------------------------------------------- one (sequence, layer)

class Unit:
    """The cache of one (sequence, layer): QEvict §4.3 Eq. (2), C = (S, L_t, F_t, Q_t, E_t)."""

    def __init__(self, cfg: Config):
        self.cfg = cfg
        self.bud = budget(cfg)
        ncap = cfg.n_windows_cap()
        self.T = 0
        self.n_route = 0                       # windows routed so far (ids below it left L_t)
        self.sink_k = self.sink_v = None       # [n_s][H_kv][d]
        self.local: Dict[int, Tuple[np.ndarray, np.ndarray]] = {}   # position -> (k, v) [H_kv][d]
        self.z = np.full(ncap, LOCAL, np.int8)
        self.S = np.zeros(ncap, np.float64)    # cumulative score, QEvict §4.2 Eq. (1)
        self.U = np.zeros(ncap, np.float64)    # attention since the previous routing event, App. J Eq. (20)
        self.R = np.zeros(ncap, np.float64)    # the ranker's value of every window (App. J)
        self.full: Dict[int, Tuple[np.ndarray, np.ndarray]] = {}    # wid -> (K, V) [W][H_kv][d]
        self.ledger: Dict[int, Ledger] = {}
        self.f_slot: Dict[int, int] = {}
        self.counters = np.zeros(len(COUNTER_NAMES), np.int64)
        self.last_transitions: Dict[str, List[int]] = {}
        self.rope: Optional[np.ndarray] = None   # [positions][64][2] (cos, sin), an input

    def set_rope_table(self, table: np.ndarray) -> None:
        self.rope = np.asarray(table, np.float32)

    def window_cs(self, w: int) -> Optional[np.ndarray]:
        """(cos, sin) rows of window w's positions, or None when keys carry no rotation."""
        if self.cfg.rope_base <= 0:
            return None
        assert self.rope is not None, "rope_base > 0 needs a rotation table"
        lo = self.cfg.n_sink + w * self.cfg.window
        return self.rope[lo:lo + self.cfg.window]

    # ---- prefill (QEvict §4.2 last paragraph; §4.3 Eq. (2))
    def prefill_route(self, k: np.ndarray, v: np.ndarray, s0: np.ndarray):
        """Prompt k, v [P][H_kv][d] (bf16 values); s0: initial scores of the prompt's windows."""
        cfg = self.cfg
        P = k.shape[0]
        assert P == cfg.prompt_len and P >= cfg.n_sink
        k = np.asarray(k, np.float32)
        v = np.asarray(v, np.float32)
        self.sink_k, self.sink_v = k[:cfg.n_sink].copy(), v[:cfg.n_sink].copy()
        for p in range(cfg.n_sink, P):
            self.local[p] = (k[p].copy(), v[p].copy())
        self.T = P
        s0 = np.asarray(s0, np.float64)
        assert len(s0) == prompt_windows(cfg), "one initial score per window that starts in the prompt"
        self.S[:len(s0)] = s0
        self.U[:len(s0)] = s0                  # the prompt's attention is the first event's u
        self.route()

    # ---- one decode step (QEvict §4.1 attention; §4.2 Eq. (1) score accumulation)
    def accessible(self):
        """Accessible tokens in chronological order: K, V [N][H_kv][d] and window id per token (-1 = sink)."""
        cfg = self.cfg
        Ks, Vs, wid = [self.sink_k], [self.sink_v], [np.full(cfg.n_sink, -1)]
        for w in range(self.n_route):
            if self.z[w] == FULL:
                Kw, Vw = self.full[w]
            elif self.z[w] == QUANT:
                Kw, Vw = self.ledger[w].dequantize(self.window_cs(w))
            else:
                continue
            Ks.append(Kw)
            Vs.append(Vw)
            wid.append(np.full(cfg.window, w))
        pos = sorted(self.local)
        if pos:
            Ks.append(np.stack([self.local[p][0] for p in pos]))
            Vs.append(np.stack([self.local[p][1] for p in pos]))
            wid.append(np.array([window_of(p, cfg) for p in pos]))
        return np.concatenate(Ks), np.concatenate(Vs), np.concatenate(wid)

    def decode_step(self, q: np.ndarray, k_new: np.ndarray, v_new: np.ndarray):
        """Append (k_new, v_new) at position T, attend with q [H_q][d] over the accessible set.

        Reading: the new token attends to itself (append, then attend).  Every
        non-sink accessible window accumulates its mass into S, including windows
        still in the recent region, so aged windows enter the pool with a score.
        Returns o [H_q][d] (float64), per-head window masses [H_q][n_cap] and per-head sink mass.
        """
        cfg = self.cfg
        self.local[self.T] = (np.asarray(k_new, np.float32).copy(), np.asarray(v_new, np.float32).copy())
        self.T += 1
        K, V, wid = self.accessible()
        o, a = attend(q, K, V, cfg.h_kv)
        ncap = len(self.S)
        masses = np.zeros((cfg.h_q, ncap))
        hist = wid >= 0
        for h in range(cfg.h_q):
            masses[h] = np.bincount(wid[hist], weights=a[h, hist], minlength=ncap)[:ncap]
        sink_mass = a[:, ~hist].sum(axis=1)
        self.S += masses.sum(axis=0) / cfg.h_q
        self.U += masses.sum(axis=0) / cfg.h_q
        return o, masses, sink_mass

    def key_norm(self, w: int) -> float:
        """Mean L2 norm of the window's cached keys, each token's key over all KV heads (App. J Eq. (24)
        up to the sign, which becomes an ascending ranking)."""
        cfg = self.cfg
        lo = cfg.n_sink + w * cfg.window
        return float(np.mean([np.sqrt(np.sum(np.asarray(self.local[p][0], np.float64) ** 2))
                              for p in range(lo, lo + cfg.window)]))

    def rank_values(self, cand: List[int], aged: List[int]) -> None:
        """Fold the event's attention u = U into the ranker's value R (App. J), then reset U."""
        cfg = self.cfg
        if cfg.ranker == 0:      # cumulative, Eq. (21): S already holds S_prev + u
            self.R[:] = self.S
        elif cfg.ranker == 1:    # decayed, Eq. (22)
            self.R[:] = cfg.decay * self.R + self.U
        elif cfg.ranker == 2:    # p-norm, Eq. (23): ranked by sum_r u_r^p, the same order as its p-th root
            self.R[:] = self.R + self.U ** cfg.pnorm
        else:                    # key norm, Eq. (24): computed once, when the window leaves the recent region
            for w in aged:
                self.R[w] = self.key_norm(w)
        self.U[:] = 0.0

    # ---- routing event (QEvict §4.3 Eq. (4)-(6), App. A Algorithm 1)
    def route(self, scores: Optional[np.ndarray] = None, rank_hook=None):
        """Route at the current T.  `scores` overrides S (the "identical scores" parity mode).

        Candidates (Eq. (4)): windows now Full or Quantized plus the windows aged
        since the last event; Evicted windows never return (Eq. (6)).
        Ranking (Eq. (5)): by score, descending; ties by window id ascending (the
        older window first, a reading: the pages do not order ties).  The first
        K_f become Full, the next K_q Quantized, the rest Evicted.
        """
        cfg, bud = self.cfg, self.bud
        n_new = n_hist(self.T, cfg)
        aged = list(range(self.n_route, n_new))
        prev = {w: int(self.z[w]) for w in range(self.n_route) if self.z[w] in (FULL, QUANT)}
        cand = sorted(list(prev) + aged)
        self.rank_values(cand, aged)
        if rank_hook is not None:                # lets a parity test compare the rank values first
            rank_hook(self.R)
        if scores is not None:                   # the "identical scores" parity mode: rank on these
            self.R[:len(scores)] = np.asarray(scores, np.float64)
            if cfg.ranker == 0:
                self.S[:len(scores)] = np.asarray(scores, np.float64)
        if cfg.ranker == 3:                      # lower key norms first (Eq. (24)'s negative sign)
            order = sorted(cand, key=lambda w: (float(self.R[w]), w))
        else:
            order = sorted(cand, key=lambda w: (-float(self.R[w]), w))
        if cfg.no_promotion:
            # App. K: a quantized window cannot return to the full tier, so the full tier takes the
            # best-ranked candidates that are not quantized; the quantized tier the next best of the rest
            new_f = set([w for w in order if prev.get(w) != QUANT][:bud.k_f])
            rest = [w for w in order if w not in new_f]
            new_q = set(rest[:bud.k_q])
            new_e = set(rest[bud.k_q:])
        else:
            new_f = set(order[:bud.k_f])
            new_q = set(order[bud.k_f:bud.k_f + bud.k_q])
            new_e = set(order[bud.k_f + bud.k_q:])
        ctr = dict.fromkeys(COUNTER_NAMES, 0)
        tr = {"promote": [], "demote": [], "quantize": [], "reactivate": [], "evict": [],
              "aged_full": [], "aged_quant": []}
        window_data = {}                         # sources read before any slot is reused

        def window_tokens(w):
            lo = cfg.n_sink + w * cfg.window
            return (np.stack([self.local[p][0] for p in range(lo, lo + cfg.window)]),
                    np.stack([self.local[p][1] for p in range(lo, lo + cfg.window)]))

        for w in aged:
            window_data[w] = window_tokens(w)
        # releases first (Algorithm 1: release evicted windows, drop their ledgers)
        for w in sorted(new_e):
            self.f_slot.pop(w, None)
            self.full.pop(w, None)
            self.ledger.pop(w, None)
            self.z[w] = EVICTED
            ctr["evictions"] += 1
            tr["evict"].append(w)
        # Quantized tier (Algorithm 1: quantise once / reactivate a dormant ledger)
        need_ledger = []
        for w in sorted(new_q):
            was = prev.get(w)
            if was == QUANT:
                continue
            if was == FULL:
                ctr["demotions"] += 1
                tr["demote"].append(w)
                src = self.full.pop(w)
                self.f_slot.pop(w)
                if w in self.ledger:
                    self.ledger[w].status = ACTIVE
                    ctr["reactivations"] += 1
                    tr["reactivate"].append(w)
                else:
                    self.ledger[w] = quantize_window(src[0], src[1], cfg.bits, self.window_cs(w))
                    need_ledger.append(w)
                    ctr["first_quant"] += 1
                    tr["quantize"].append(w)
            else:                                  # aged straight into the quantized tier
                self.ledger[w] = quantize_window(*window_data[w], cfg.bits, self.window_cs(w))
                need_ledger.append(w)
                ctr["first_quant"] += 1
                ctr["aged_quant"] += 1
                tr["quantize"].append(w)
                tr["aged_quant"].append(w)
            self.z[w] = QUANT
        # Full tier (Algorithm 1: a promoted window is rebuilt from its ledger, which turns dormant)
        need_fslot = []
        for w in sorted(new_f):
            was = prev.get(w)
            if was == FULL:
                continue
            if was == QUANT:
                led = self.ledger[w]
                self.full[w] = led.dequantize(self.window_cs(w))
                led.status = DORMANT
                ctr["promotions"] += 1
                tr["promote"].append(w)
            else:
                self.full[w] = window_data[w]
                ctr["aged_full"] += 1
                tr["aged_full"].append(w)
            need_fslot.append(w)
            self.z[w] = FULL
        # deterministic slots: after the releases, requests in ascending window id take the
        # lowest free indices (F pool of K_f slots, ledger pool of K_f + K_q slots)
        used_f = set(self.f_slot.values())
        free_f = [s for s in range(bud.k_f) if s not in used_f]
        for i, w in enumerate(need_fslot):
            self.f_slot[w] = free_f[i]
        used_l = {led.slot for ww, led in self.ledger.items() if ww not in need_ledger}
        free_l = [s for s in range(bud.k_f + bud.k_q) if s not in used_l]
        for i, w in enumerate(need_ledger):
            self.ledger[w].slot = free_l[i]
        for w in aged:                                  # aged windows leave the recent region
            lo = cfg.n_sink + w * cfg.window
            for p in range(lo, lo + cfg.window):
                del self.local[p]
        self.n_route = n_new
        self.counters += np.array([ctr[n] for n in COUNTER_NAMES], np.int64)
        self.last_transitions = tr
        return ctr

    # ---- views used by the parity tests
    def f_table(self) -> List[Tuple[int, int]]:
        return sorted((w, s) for w, s in self.f_slot.items())

    def q_table(self) -> List[Tuple[int, int]]:
        return sorted((w, led.slot) for w, led in self.ledger.items() if led.status == ACTIVE)

    def ledger_status(self) -> np.ndarray:
        st = np.zeros(len(self.z), np.int8)
        for w, led in self.ledger.items():
            st[w] = led.status
        return st

    def stored_bytes(self) -> int:
        """Persistent bytes charged to the budget (QEvict App. B.4 Eq. (8)) at this moment."""
        bud = self.bud
        nf = sum(1 for w in range(self.n_route) if self.z[w] == FULL)
        nq = sum(1 for w in range(self.n_route) if self.z[w] == QUANT)
        return bud.b_sink + bud.b_local + nf * bud.m_f + nq * bud.m_q
