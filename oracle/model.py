"""Oracle: one decode step of the DeepSeek-V2-style OCR text decoder, float64.

TEST INFRASTRUCTURE.  Only tests/, __graft_entry__.smoke() and bench.py's
cpu_baseline / reference leg may import anything under oracle/.  It shares no
code with the CUDA library and never imports it.

Every row is processed on its own, in textbook order, in float64, except
that the activations the method stores in fp16 are rounded to fp16 (round to
nearest even) where it stores them: the normalised inputs of the matmuls
(before QKV, the router and experts / MLP, and the LM head), the keys and
values written to the KV cache, the attention output, and the SwiGLU
activations.  The residual stream, accumulations, RoPE, softmax, logits and
routing weights stay float64.  Inputs that the workload fixes in fp16
(embeddings, hidden inputs, cached keys/values, norm weights) are read
exactly as given.

Sources, by page and section:

* "Unlimited-OCR on Apple Silicon with C and Metal",
  - "Il decoder e il Mixture of Experts": 12 layers, 10 heads x 128, the first
    layer a dense MLP, the next 11 MoE with 64 routed experts, top-6, two
    shared experts; route, group tokens by expert, run, recompose; the decode
    loop appends to the KV cache and ends in an argmax over the language head;
    generated tokens live in a 128-token ring buffer.
  - "Quantizzazione: Q8 prima, Q4 dove conviene": dequantisation inside the
    matmul kernels; norms and activations stay fp16.
* "Falcon-OCR INT8 OpenVINO IR" model card, intro: the attention sink is one
  extra key whose logit is the sink and whose value is zero, equivalent to
  rescaling the output by sigmoid(lse - sink); the KV cache is an input the
  step writes in place.

Readings where the pages are silent (also listed in the design notes):
RMSNorm x / sqrt(mean(x^2) + eps) * w; rotate-half RoPE with theta 10000 at
the absolute position, applied to q and k before caching; plain multi-head
attention with scale 1/sqrt(D); SwiGLU experts down(silu(gate x) * up x);
top-k chosen on router logits (lowest index wins a tie), weights =
softmax probabilities renormalised over the chosen k; shared experts with
weight 1; the sink logit enters the softmax unscaled; greedy argmax takes the
lowest index among equal maxima.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

from .quant import dequant, float32_is_exact, F16

# tensor kinds of the canonical weight list (the C header's enumeration)
T_EMBED, T_FINAL_NORM, T_LM_HEAD = 0, 1, 2
T_ATTN_NORM, T_WQ, T_WK, T_WV, T_WO, T_MLP_NORM = 3, 4, 5, 6, 7, 8
T_GATE, T_UP, T_DOWN = 9, 10, 11
T_ROUTER = 12
T_SHARED_GATE, T_SHARED_UP, T_SHARED_DOWN = 13, 14, 15
T_EXPERT_GATE, T_EXPERT_UP, T_EXPERT_DOWN = 16, 17, 18
T_PROJ, T_PROJ_BIAS = 19, 20


# ------------------------------------------------------------------ primitives
def f16(x):
    """Round to fp16 (nearest even), as the method stores an activation; float64 result."""
    return np.asarray(x, dtype=np.float64).astype(np.float16).astype(np.float64)


def rmsnorm(x, w, eps):
    """x / sqrt(mean(x^2) + eps) * w over the last axis (Metal page: norms)."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * w


def silu(z):
    return z / (1.0 + np.exp(-z))


def swiglu(x, wg, wu, wd):
    """One gated expert / dense MLP: down(silu(gate x) * up x)."""
    return wd @ (silu(wg @ x) * (wu @ x))


def swiglu_rows(X, wg, wu, wd, act_fp16=False):
    """swiglu applied to every row of X (one matmul per projection); with
    act_fp16 the activations silu(gate x) * up x are stored in fp16 before the
    down projection, as the method stores them."""
    a = silu(X @ wg.T) * (X @ wu.T)
    return (f16(a) if act_fp16 else a) @ wd.T


def rope(v, pos, theta):
    """Rotate-half rotary embedding of v[..., D] at absolute position pos.

    Pair (i, i + D/2) turns by the angle pos * theta^(-2i/D).
    """
    D = v.shape[-1]
    half = D // 2
    inv_freq = theta ** (-(2.0 * np.arange(half)) / D)
    ang = pos * inv_freq
    c, s = np.cos(ang), np.sin(ang)
    a, b = v[..., :half], v[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def kv_quant(x):
    """INT8 KV cache entry of key or value vectors (last axis = one head's D values).

    Symmetric, one scale per vector: s = max|x| / 127, code = round(x / s)
    (half to even) clamped to [-127, 127]; a zero vector has s = 0 and zero
    codes.  The scale and the codes are integer decisions taken in floating
    point, so they are taken in fp32, the precision the kernels store and
    divide in ("Falcon-OCR INT8 OpenVINO IR", "How it is meant to be run": the
    service keeps an INT8 KV cache; the per-head scale is this reading).
    Returns (codes int8 [..., D], s float32 [...]).
    """
    x = np.asarray(x, dtype=np.float64).astype(np.float32)
    amax = np.max(np.abs(x), axis=-1)
    s = (amax / np.float32(127.0)).astype(np.float32)
    safe = np.where(s > 0, s, np.float32(1.0)).astype(np.float32)
    q = np.rint((x / safe[..., None]).astype(np.float32))
    q = np.where(s[..., None] > 0, np.clip(q, -127, 127), 0)
    return q.astype(np.int8), s


def act_quant(x, group=32):
    """Dynamic int8 quantisation of projection inputs, per group of `group`
    consecutive inputs (last axis): the same symmetric rule as kv_quant per
    group (s = max|x| / 127, code = round-half-even(x / s), fp32 decisions).
    Returns the quantised values s * code (float64), the ones the projection
    multiplies ("Falcon-OCR INT8 OpenVINO IR": the runtime quantises the linear
    layers' inputs dynamically in groups of 32, src_dyn_quant_group_size:32).
    """
    x = np.asarray(x, dtype=np.float64)
    shape = x.shape
    g = x.reshape(shape[:-1] + (shape[-1] // group, group))
    codes, s = kv_quant(g)
    return kv_dequant(codes, s).reshape(shape)


def kv_dequant(codes, s):
    """Value of an INT8 KV entry: s * code (float64)."""
    return np.asarray(codes, dtype=np.float64) * np.asarray(s, dtype=np.float64)[..., None]


def project(feats, W, b=None):
    """The projector that takes visual features into the decoder's hidden space:
    y = W x (+ b), stored in fp16 as the decoder's input embeddings.

    "Unlimited-OCR on Apple Silicon with C and Metal", "Il modello: una
    pipeline vision-language completa" (the two encoders' features pass through
    a projector from 2048 to 1280 dimensions) and "Quantizzazione" (the Q8
    profile covers the projector; biases stay fp16).  A single linear map with
    a bias is the reading taken.
    """
    y = np.asarray(feats, dtype=np.float64) @ W.T
    if b is not None:
        y = y + b
    return f16(y)


def ring_slot(p, P, R):
    """Cache slot of absolute position p: prefix slots 0..P-1, then a ring of R."""
    return p if p < P else P + (p - P) % R


def attend(q, K, V, sink=None):
    """softmax(K q / sqrt(D)) V over the given keys, optionally with a sink key.

    The sink is one more logit (unscaled) whose value vector is zero
    (Falcon-OCR page, intro).
    """
    D = q.shape[-1]
    s = (K @ q) / math.sqrt(D)
    m = s.max()
    if sink is not None:
        m = max(m, sink)
    e = np.exp(s - m)
    z = e.sum()
    if sink is not None:
        z += math.exp(sink - m)
    return (e @ V) / z


def attend_lse(q, K, V):
    """Plain attention output and its log-sum-exp of scaled logits."""
    D = q.shape[-1]
    s = (K @ q) / math.sqrt(D)
    m = s.max()
    e = np.exp(s - m)
    return (e @ V) / e.sum(), m + math.log(e.sum())


def route(logits, k):
    """Softmax over the router logits, top-k by logit, renormalised weights.

    Selection is on the logits (softmax is monotone); ties go to the lower
    expert index.  Returns (idx[k], w[k]).
    """
    logits = np.asarray(logits, dtype=np.float64)
    p = np.exp(logits - logits.max())
    p /= p.sum()
    order = np.argsort(-logits, kind="stable")
    idx = order[:k]
    w = p[idx] / p[idx].sum()
    return idx.astype(np.int64), w


# Logit gap under which a selection on logits is not decided by the definition
# alone.  The decode-step statement fixes 1e-2 as the top-2 margin below which
# greedy ids may differ; the router's top-k is the step's other selection on
# logits, so its k-th vs (k+1)-th gap takes the same margin: below it another
# set is an equally correct top-k for a computation within the float tolerance.
TIE_TOL = 1e-2


def group_by_expert(idx, n_experts):
    """Histogram, exclusive scan and expert-grouped permutation of (row, slot).

    perm lists the entries row*k + slot grouped by expert ascending, rows
    ascending within an expert.  (Metal page: group the tokens by expert.)
    """
    idx = np.asarray(idx)
    rows, k = idx.shape
    count = np.zeros(n_experts, dtype=np.int64)
    for r in range(rows):
        for s in range(k):
            count[idx[r, s]] += 1
    offset = np.zeros(n_experts + 1, dtype=np.int64)
    for e in range(n_experts):
        offset[e + 1] = offset[e] + count[e]
    perm = np.zeros(rows * k, dtype=np.int64)
    fill = offset[:-1].copy()
    for e in range(n_experts):
        for r in range(rows):
            for s in range(k):
                if idx[r, s] == e:
                    perm[fill[e]] = r * k + s
                    fill[e] += 1
    return count, offset, perm


def argmax_first(v):
    """Index of the first maximum (greedy decode, lowest index on ties)."""
    return int(np.argmax(v))


# ------------------------------------------------------------------ model
@dataclass
class StepResult:
    hidden: np.ndarray          # [L+1, rows, H]: input of layer 0, output of each layer
    h_attn: np.ndarray          # [L, rows, H]: residual after attention
    k_new: np.ndarray           # [L, rows, nh, D] keys written this step (after RoPE)
    v_new: np.ndarray           # [L, rows, nh, D]
    slots: np.ndarray           # [rows] cache slot written this step
    router: dict = field(default_factory=dict)   # layer -> dict(logits, idx, w, count, offset, perm)
    logits: np.ndarray | None = None   # [rows, V]
    next_ids: np.ndarray | None = None  # [rows]
    margin: np.ndarray | None = None    # [rows] top-1 minus top-2 logit
    kv_entries: dict | None = None      # INT8 cache: layer -> (k codes, k scales, v codes, v scales) [rows][nh]..


class OracleModel:
    """Float64 decode-step model over the canonical weight list.

    cfg: any object with the model-config attributes (hidden, n_heads,
    head_dim, n_layers, n_dense_layers, dense_inter, n_experts, top_k,
    n_shared, expert_inter, vocab, prefix_len, ring_len, use_sink, rms_eps,
    rope_theta).
    tensors: objects with kind, layer, expert, fmt, rows, cols, blob.
    kv_prefix: optional list over layers of (k, v) fp16 [rows, nh, P, D]
    (a cached prefix); without it the prefix is filled by decode steps.
    sinks: optional fp32 [layers, heads].
    kv_int8: the KV cache holds INT8 entries (kv_quant) instead of fp16 values:
    every key and value vector is quantised when it is written (the cached
    prefix included) and attention reads s * code.
    """

    def __init__(self, cfg, tensors, rows, kv_prefix=None, sinks=None, cache="float64", kv_int8=False,
                 act_int8=False):
        self.cfg = cfg
        self.rows = rows
        self.kv_int8 = kv_int8
        # dynamic int8 activations: the inputs of the dense projections (Q/K/V, O,
        # dense gate/up and down) are quantised per group of 32 before the matmul
        self.act_int8 = act_int8
        self._t = {(t.kind, t.layer, t.expert): t for t in tensors}
        # cache: None (dequantise at every use), "float64", or "float32" (only
        # for matrices whose values are exact in float32, see quant.float32_is_exact)
        self._cache = {} if cache else None
        self._cache_dtype = cache
        self.sinks = None if sinks is None else np.asarray(sinks, dtype=np.float64)
        nh, D, P, R, L = cfg.n_heads, cfg.head_dim, cfg.prefix_len, cfg.ring_len, cfg.n_layers
        self.P, self.R = P, R
        # per layer: prefix keys/values [rows, nh, P, D] and ring [rows, nh, R, D]
        self.pk, self.pv = [], []
        for l in range(L):
            if kv_prefix is not None:
                k, v = kv_prefix[l]
                if kv_int8:
                    k, v = kv_dequant(*kv_quant(k)), kv_dequant(*kv_quant(v))
                self.pk.append(k)
                self.pv.append(v)
            else:
                self.pk.append(np.zeros((rows, nh, P, D)))
                self.pv.append(np.zeros((rows, nh, P, D)))
        self.rk = [np.zeros((rows, nh, R, D)) for _ in range(L)]
        self.rv = [np.zeros((rows, nh, R, D)) for _ in range(L)]
        # absolute position held by each slot (-1: never written); same for all layers
        self.slot_pos = np.full((rows, P + R), -1, dtype=np.int64)
        if kv_prefix is not None:
            self.slot_pos[:, :P] = np.arange(P)

    # ---------------------------------------------------------------- weights
    def w(self, kind, layer=0, expert=0):
        key = (kind, layer, expert)
        if self._cache is not None and key in self._cache:
            return np.asarray(self._cache[key], dtype=np.float64)
        t = self._t[key]
        m = dequant(t.blob, t.fmt, t.rows, t.cols)
        if t.rows == 1:
            m = m[0]
        if self._cache is not None:
            if self._cache_dtype == "float32" and float32_is_exact(m):
                self._cache[key] = m.astype(np.float32)
            else:
                self._cache[key] = m
        return m

    # ---------------------------------------------------------------- projector
    def project(self, feats):
        """Visual features [n, proj_in] -> fp16 embeddings [n, hidden]."""
        b = self.w(T_PROJ_BIAS) if (T_PROJ_BIAS, 0, 0) in self._t else None
        return project(feats, self.w(T_PROJ), b)

    # ---------------------------------------------------------------- attention
    def _valid(self, row, p):
        """Slots whose stored position q satisfies q <= p and (q < P or q > p - R)."""
        q = self.slot_pos[row]
        return (q >= 0) & (q <= p) & ((q < self.P) | (q > p - self.R))

    def _attention(self, layer, row, qh, p):
        cfg = self.cfg
        valid = self._valid(row, p)
        vp, vr = valid[: self.P], valid[self.P:]
        out = np.zeros((cfg.n_heads, cfg.head_dim))
        for h in range(cfg.n_heads):
            K = np.concatenate([np.asarray(self.pk[layer][row, h], dtype=np.float64)[vp],
                                self.rk[layer][row, h][vr]])
            V = np.concatenate([np.asarray(self.pv[layer][row, h], dtype=np.float64)[vp],
                                self.rv[layer][row, h][vr]])
            sink = None
            if cfg.use_sink:
                sink = float(self.sinks[layer, h])
            out[h] = attend(qh[h], K, V, sink)
        return out

    # ---------------------------------------------------------------- step
    def step(self, positions, ids=None, x=None, want_logits=True):
        """One decode step for every row.

        positions: int [rows]; ids: int [rows] token ids (embedding lookup) or
        x: fp16 [rows, H] hidden inputs.
        """
        cfg = self.cfg
        rows, H, nh, D, L = self.rows, cfg.hidden, cfg.n_heads, cfg.head_dim, cfg.n_layers
        positions = np.asarray(positions, dtype=np.int64)
        if x is None:
            emb = self.w(T_EMBED)
            X = np.stack([emb[int(i)] for i in ids])
        else:
            X = np.asarray(x, dtype=np.float64).reshape(rows, H)
        res = StepResult(hidden=np.zeros((L + 1, rows, H)), h_attn=np.zeros((L, rows, H)),
                         k_new=np.zeros((L, rows, nh, D)), v_new=np.zeros((L, rows, nh, D)),
                         slots=np.array([ring_slot(int(p), self.P, self.R) for p in positions]))
        res.hidden[0] = X
        for r in range(rows):
            self.slot_pos[r, res.slots[r]] = positions[r]
        aq = act_quant if self.act_int8 else (lambda v: v)
        for l in range(L):
            Xn = aq(f16(rmsnorm(X, self.w(T_ATTN_NORM, l), cfg.rms_eps)))
            Q = Xn @ self.w(T_WQ, l).T
            Kx = Xn @ self.w(T_WK, l).T
            Vx = Xn @ self.w(T_WV, l).T
            attn = np.zeros((rows, nh * D))
            for r in range(rows):
                p = int(positions[r])
                qh = rope(Q[r].reshape(nh, D), p, cfg.rope_theta)
                if self.kv_int8:  # the cache holds INT8 entries, one scale per head
                    kq = kv_quant(rope(Kx[r].reshape(nh, D), p, cfg.rope_theta))
                    vq = kv_quant(Vx[r].reshape(nh, D))
                    kh, vh = kv_dequant(*kq), kv_dequant(*vq)
                    if res.kv_entries is None:
                        res.kv_entries = {}
                    res.kv_entries.setdefault(l, []).append((kq[0], kq[1], vq[0], vq[1]))
                else:  # the cache holds fp16
                    kh = f16(rope(Kx[r].reshape(nh, D), p, cfg.rope_theta))
                    vh = f16(Vx[r].reshape(nh, D))
                res.k_new[l, r], res.v_new[l, r] = kh, vh
                s = int(res.slots[r])
                if s < self.P:
                    self.pk[l][r, :, s] = kh
                    self.pv[l][r, :, s] = vh
                else:
                    self.rk[l][r, :, s - self.P] = kh
                    self.rv[l][r, :, s - self.P] = vh
                attn[r] = f16(self._attention(l, r, qh, p).reshape(-1))
            Hh = X + aq(attn) @ self.w(T_WO, l).T
            res.h_attn[l] = Hh
            Hn = f16(rmsnorm(Hh, self.w(T_MLP_NORM, l), cfg.rms_eps))
            if l < cfg.n_dense_layers or cfg.n_experts == 0:
                if self.act_int8:
                    a = f16(silu(aq(Hn) @ self.w(T_GATE, l).T) * (aq(Hn) @ self.w(T_UP, l).T))
                    Y = Hh + aq(a) @ self.w(T_DOWN, l).T
                else:
                    Y = Hh + swiglu_rows(Hn, self.w(T_GATE, l), self.w(T_UP, l), self.w(T_DOWN, l), act_fp16=True)
            else:
                Y, info = self._moe(l, Hh, Hn)
                res.router[l] = info
            res.hidden[l + 1] = Y
            X = Y
        if cfg.vocab and want_logits:
            Xn = f16(rmsnorm(X, self.w(T_FINAL_NORM), cfg.rms_eps))
            logits = Xn @ self.w(T_LM_HEAD).T
            res.logits = logits
            res.next_ids = np.array([argmax_first(logits[r]) for r in range(rows)])
            top2 = np.sort(logits, axis=-1)[:, -2:]
            res.margin = top2[:, 1] - top2[:, 0]
        return res

    def _moe(self, l, Hh, Hn):
        """Router, top-k, weighted routed experts plus shared experts, residual.

        Each expert is applied to all the rows that selected it with one
        matmul; row r's result is still exactly sum_j w_rj * E_j(x_r).
        """
        cfg = self.cfg
        rows, k, E = self.rows, cfg.top_k, cfg.n_experts
        Wr = self.w(T_ROUTER, l)
        logits = Hn @ Wr.T
        # the k-th vs (k+1)-th logit gap decides whether the selected set is well defined
        srt = np.sort(logits, axis=-1)[:, ::-1]
        gap = srt[:, k - 1] - srt[:, k] if k < E else np.full(rows, np.inf)
        idx = np.zeros((rows, k), dtype=np.int64)
        wts = np.zeros((rows, k))
        for r in range(rows):
            idx[r], wts[r] = route(logits[r], k)
        Y = Hh.copy()
        for e in range(E):
            sel_r, sel_j = np.nonzero(idx == e)
            if sel_r.size == 0:
                continue
            out = swiglu_rows(Hn[sel_r], self.w(T_EXPERT_GATE, l, e), self.w(T_EXPERT_UP, l, e),
                              self.w(T_EXPERT_DOWN, l, e), act_fp16=True)
            for i in range(sel_r.size):
                Y[sel_r[i]] += wts[sel_r[i], sel_j[i]] * out[i]
        for s in range(cfg.n_shared):
            Y += swiglu_rows(Hn, self.w(T_SHARED_GATE, l, s), self.w(T_SHARED_UP, l, s),
                             self.w(T_SHARED_DOWN, l, s), act_fp16=True)
        count, offset, perm = group_by_expert(idx, E)
        return Y, dict(logits=logits, idx=idx, w=wts, count=count, offset=offset,
                       perm=perm, gap=gap)
