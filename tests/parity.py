"""Free-running parity of the CUDA library (through the C ABI) against the oracle.

Both sides consume the same seeded workload; nothing the library computes is
ever an input of the oracle.  For token-id workloads the library is fed the
oracle's greedy ids (teacher forcing by the oracle), so a near-tie argmax
cannot make the two inputs diverge.

Comparison rules (the decode-step statement's tolerances):
* every floating-point output (hidden state after attention and after each
  layer, the K and V written to the cache, router logits, LM logits):
  relative L2 error <= 2e-3 and max abs error <= 2e-2 against the oracle;
* integer outputs bit-exact: the router's top-k set where the oracle's k-th
  vs (k+1)-th logit gap exceeds a fixed gate (1e-2, the margin the statement
  gives for a selection on logits; 1e-3 where the router's inputs coincide),
  argmax ids where the oracle's top-2 margin exceeds 1e-2, the grouping
  (count / offset / permutation equal to the stable grouping of the
  library's own top-k, and each compared row's (row, expert) entries equal
  to the oracle's); the library's set is always exactly the top-k of its own
  fp32 logits;
* routing weights: equal (rel-L2 1e-5) to the float64 softmax of the
  library's own logits renormalised over its own set, and against the oracle
  at rel-L2 2e-3 wherever the router's inputs coincide on both sides (single
  layers fed the same hidden vectors).  Deeper in a free-running stack the
  fp16 activations of the two sides drift apart by up to the float tolerance,
  which moves every router logit by up to d = max|logit difference|; the
  renormalised softmax turns that into a relative weight error of at most
  2 d (to first order: dw_i = w_i (dl_i - sum_j w_j dl_j)), so there the
  weights are held to max(2e-3, 2 d) with the logits themselves at the
  stated tolerance;
* dynamic int8 activations (the Falcon-OCR card's groups of 32): both sides
  take the code decisions in fp32, but on inputs that agree only to rounding
  (fp16 activations of an fp32 and a float64 residual stream), so an input
  near a rounding boundary of the code grid can land one code step apart.  One
  step moves the projection by s * w (s = group max / 127): a full grid step,
  sqrt(12) times the rms error the grid itself adds per input.  Two correct
  quantisers whose inputs differ by less than a step disagree by at most one
  step on every code, which moves the output by at most about sqrt(12) * eps_q,
  with eps_q = (group max / rms) / (127 sqrt 12) ~ 0.5-0.7% the grid's own
  relative error on these activations: ~2e-2 (the differences grow with depth
  as the two sides' inputs drift; 18 int8-asym layers reach 1.1e-2).  So int8-
  activation runs hold every vector to rel-L2 <= 2e-2 and max-abs <= 0.2 (the
  stated pair scaled by the same factor 10: a code step moves every element of
  the output, so the largest element error grows with the rms one) and the
  median rel-L2 over all compared vectors to the plain 2e-3; a wrong scale,
  zero point or k order errs by tens of percent;
* a router set that differs at a near tie is counted, not failed; it changes
  that row's layer output, so the rest of the row's layers at that step are
  not compared, and before the next step the library's cache entries of the
  layers above are overwritten with the oracle's (the library takes the
  oracle's state; the oracle never takes the library's).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

import oracle

REL_L2 = 2e-3
REL_L2_INT8_ACT = 2e-2  # per vector with int8 activations: every code one step apart (median still <= REL_L2)
MAX_ABS_INT8_ACT = 0.2  # ... and max-abs, the stated pair scaled by the same factor
_active_rel = [REL_L2]  # the per-vector bound of the run in progress
_active_abs = [0.0]     # its max-abs bound (set with it)
oracle_kv_quant = oracle.kv_quant  # entries of values the oracle's INT8 cache holds (scale * code: idempotent)
MAX_ABS = 2e-2
ROUTER_GAP = oracle.TIE_TOL  # router sets are compared where the oracle's gap exceeds it
ROUTER_GAP_SAME_INPUT = 1e-3  # ... and where the router's inputs coincide on both sides
ID_MARGIN = 1e-2
OWN_WEIGHTS_REL = 1e-5  # the library's weights against the softmax of its own logits


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def check_close(name, got, want, rel=None, mx=None):
    rel = _active_rel[0] if rel is None else rel
    mx = (_active_abs[0] or MAX_ABS) if mx is None else mx
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert got.shape == want.shape, (name, got.shape, want.shape)
    e = rel_l2(got, want)
    m = float(np.max(np.abs(got - want))) if got.size else 0.0
    assert e <= rel and m <= mx, f"{name}: rel-L2 {e:.3e} (<= {rel}), max-abs {m:.3e} (<= {mx})"
    return e, m, name


@dataclass
class Stats:
    steps: int = 0
    float_checks: int = 0
    worst_rel: float = 0.0
    worst_abs: float = 0.0
    router_checks: int = 0
    router_near_ties: int = 0
    id_checks: int = 0
    id_near_ties: int = 0
    kv_checks: int = 0
    kv_codes: int = 0          # INT8 cache codes compared
    kv_code_steps: int = 0     # ... that differ from the oracle's by one step
    grouping_checks: int = 0
    worst_weights_rel: float = 0.0
    tainted_rows: set = field(default_factory=set)

    worst_name: str = ""
    rels: list = field(default_factory=list)  # rel-L2 of every compared vector

    def note(self, e, m, name=""):
        self.float_checks += 1
        self.rels.append(e)
        if e > self.worst_rel:
            self.worst_name = name
        self.worst_rel = max(self.worst_rel, e)
        self.worst_abs = max(self.worst_abs, m)


class LibraryRunner:
    """Drives one library context over a workload with torch device buffers."""

    def __init__(self, ctx, wl, rows=None):
        import torch

        self.torch = torch
        self.ctx = ctx
        self.wl = wl
        self.rows = rows or wl.rows
        cfg = wl.cfg
        dev = torch.device("cuda")
        self.pos = torch.zeros(self.rows, dtype=torch.int32, device=dev)
        self.ids = torch.zeros(self.rows, dtype=torch.int32, device=dev)
        self.next = torch.zeros(self.rows, dtype=torch.int32, device=dev)
        self.x = torch.zeros((self.rows, cfg.hidden), dtype=torch.int16, device=dev)
        self.y = torch.zeros((self.rows, cfg.hidden), dtype=torch.float32, device=dev)
        self.logits = torch.zeros((self.rows, max(cfg.vocab, 1)), dtype=torch.float32, device=dev)

    def step(self, positions, ids=None, x=None, want_logits=False):
        t = self.torch
        self.pos.copy_(t.from_numpy(np.asarray(positions, np.int32)))
        lg = self.logits.data_ptr() if want_logits else 0
        if x is not None:
            self.x.copy_(t.from_numpy(np.ascontiguousarray(x, np.float16).view(np.int16)))
            nxt = self.next.data_ptr() if self.wl.cfg.vocab else 0
            self.ctx.uocr_decode_step_embeds(self.rows, self.x.data_ptr(), self.pos.data_ptr(), self.y.data_ptr(),
                                             nxt, lg)
        else:
            self.ids.copy_(t.from_numpy(np.asarray(ids, np.int32)))
            self.ctx.uocr_decode_step(self.rows, self.ids.data_ptr(), self.pos.data_ptr(), self.next.data_ptr(), lg)
        self.ctx.uocr_sync()
        out = dict(next=self.next.cpu().numpy().copy())
        if want_logits:
            out["logits"] = self.logits.cpu().numpy().copy()
        if x is not None:
            out["y"] = self.y.cpu().numpy().copy()
        return out


def own_weights(logits, idx):
    """float64 softmax of one row's logits renormalised over the chosen experts idx (in idx order)."""
    lg = np.asarray(logits, np.float64)
    e = np.exp(lg[np.asarray(idx)] - lg.max())
    return e / e.sum()


def compare_step(ctx, cfg, res, lib_rows, stats, row_map=None, check_kv=True, same_router_input=False):
    """Compare one step.  res: oracle StepResult over the oracle's rows;
    row_map[i] = library row of oracle row i.  same_router_input: the router's
    inputs are the same on both sides up to one layer of kernel rounding (a
    single layer fed hidden vectors), so weights and sets take the tight
    rules.  Returns, per oracle row, the layer whose MoE output diverged at a
    router near tie (cfg.n_layers if none)."""
    n = res.hidden.shape[1]
    row_map = list(range(n)) if row_map is None else row_map
    L = cfg.n_layers
    div = [L] * n
    taps = {}

    def tap(t):
        if t not in taps:
            taps[t] = ctx.uocr_debug_hidden(t, lib_rows)
        return taps[t]

    router_all_equal = True
    for l in range(L):
        keep = [i for i in range(n) if div[i] >= L]
        if not keep:
            break
        g = tap(2 * l)[[row_map[i] for i in keep]]
        stats.note(*check_close(f"layer {l} after attention", g, res.h_attn[l][keep]))
        if check_kv:
            for i in keep:
                r = row_map[i]
                s = int(res.slots[i])
                if cfg.kv_int8:
                    check_int8_entries(ctx.uocr_kv_read_i8(r, l, s, 1), res.kv_entries[l][i], stats,
                                       f"layer {l} row {r} slot {s}")
                    continue
                k, v = ctx.uocr_kv_read(r, l, s, 1)
                stats.note(*check_close(f"layer {l} row {r} k at slot {s}", k[:, 0].astype(np.float64),
                                        res.k_new[l, i]))
                stats.note(*check_close(f"layer {l} row {r} v at slot {s}", v[:, 0].astype(np.float64),
                                        res.v_new[l, i]))
                stats.kv_checks += 1
        out_ok = list(keep)
        if l in res.router:
            info = res.router[l]
            gr = ctx.uocr_debug_router(l, lib_rows)
            glog = ctx.uocr_debug_router_logits(l, lib_rows)
            for i in keep:
                r = row_map[i]
                want = sorted(int(e) for e in info["idx"][i])
                got = sorted(int(e) for e in gr["idx"][r])
                # the library's decision in its own precision: exactly the top-k of its fp32
                # logits, lowest index first among equal logits
                own = sorted(int(e) for e in np.argsort(-glog[r], kind="stable")[:cfg.top_k])
                assert got == own, f"layer {l} row {r}: router set {got} is not the top-k {own} of its logits"
                # router logits: a floating-point output, at the stated tolerance
                stats.note(*check_close(f"layer {l} row {r} router logits", glog[r], info["logits"][i]))
                err = float(np.max(np.abs(glog[r].astype(np.float64) - info["logits"][i])))
                # the weights are the renormalised softmax of the library's own logits
                check_close(f"layer {l} row {r} routing weights vs own logits", gr["w"][r],
                            own_weights(glog[r], gr["idx"][r]), rel=OWN_WEIGHTS_REL)
                gate = ROUTER_GAP_SAME_INPUT if same_router_input else ROUTER_GAP
                stats.router_checks += 1
                if want != got:
                    router_all_equal = False
                    assert info["gap"][i] <= gate, \
                        f"layer {l} row {r}: router set {got} != {want} with oracle gap {info['gap'][i]:.3e}"
                    stats.router_near_ties += 1
                    stats.tainted_rows.add(r)
                    out_ok.remove(i)
                    div[i] = l
                    continue
                wmap = {int(e): float(w) for e, w in zip(gr["idx"][r], gr["w"][r])}
                got_w = np.array([wmap[int(e)] for e in info["idx"][i]])
                w_rel = REL_L2 if same_router_input else max(REL_L2, 2.0 * err)
                stats.note(*check_close(f"layer {l} row {r} routing weights", got_w, info["w"][i], rel=w_rel))
                stats.worst_weights_rel = max(stats.worst_weights_rel, rel_l2(got_w, info["w"][i]))
            # grouping: unique given the top-k sets
            flat = gr["idx"].reshape(-1)
            E = cfg.n_experts
            assert np.array_equal(gr["count"], np.bincount(flat, minlength=E)), f"layer {l}: counts"
            assert np.array_equal(gr["offset"], np.concatenate([[0], np.cumsum(gr["count"])])), f"layer {l}: offsets"
            assert np.array_equal(gr["perm"], np.argsort(flat, kind="stable")), f"layer {l}: permutation"
            # unique part of the grouping: the (row, expert) entries in perm order (the
            # slot numbers inside a row depend on the order of near-equal chosen logits)
            k = cfg.top_k
            g_pairs = [(int(e) // k, int(gr["idx"][e // k][e % k])) for e in gr["perm"]]
            if router_all_equal and n == lib_rows and row_map == list(range(n)):
                assert np.array_equal(gr["count"], info["count"]), f"layer {l}: counts vs oracle"
                assert np.array_equal(gr["offset"], info["offset"]), f"layer {l}: offsets vs oracle"
                o_pairs = [(int(e) // k, int(info["idx"][e // k][e % k])) for e in info["perm"]]
                assert g_pairs == o_pairs, f"layer {l}: grouping {g_pairs} != {o_pairs}"
            for i in keep:
                # every compared row: its entries of the library's grouping, in perm order,
                # are the oracle's experts of that row in ascending order
                r = row_map[i]
                if r in stats.tainted_rows and sorted(int(e) for e in gr["idx"][r]) != \
                        sorted(int(e) for e in info["idx"][i]):
                    continue
                mine = [e for (rr, e) in g_pairs if rr == r]
                assert mine == sorted(int(e) for e in info["idx"][i]), \
                    f"layer {l} row {r}: grouping entries {mine} != oracle experts {sorted(info['idx'][i])}"
                stats.grouping_checks += 1

        if out_ok:
            g = tap(2 * l + 1)[[row_map[i] for i in out_ok]]
            stats.note(*check_close(f"layer {l} output", g, res.hidden[l + 1][out_ok]))
    return div


def check_int8_entries(got, want, stats, name, exact=False):
    """INT8 cache entries of the library (codes [nh][n][D], scales [nh][n] per
    K and V, as uocr_kv_read_i8 gives them) against the oracle's (codes
    [nh][(n,)D], scales [nh][(n)]).  The scales are floating-point outputs (the
    stated tolerance).  A code is an integer decided in floating point: where
    both sides' inputs coincide (exact) it must be equal; elsewhere the two
    sides' values differ within the float tolerance, far less than half a code
    step at the stated 2e-3, so a code may differ by one step (the rounding).
    With int8 activations the vectors agree to the int8-activation bound: the
    dequantised vectors are held to it, and an element may then be off by up
    to that bound times |x| (the vector's norm), i.e. 127 * bound * |x| / max|x|
    steps, so each head vector's codes may differ by one step more than that.
    Steps are counted."""
    gkc, gks, gvc, gvs = got
    okc, oks, ovc, ovs = want
    for nm, gc, gs, oc, os_ in (("k", gkc, gks, okc, oks), ("v", gvc, gvs, ovc, ovs)):
        gc = gc.reshape(np.asarray(oc).shape)
        gs = gs.reshape(np.asarray(os_).shape)
        stats.note(*check_close(f"{name} {nm} scales", gs, os_))
        d = np.abs(gc.astype(np.int32) - np.asarray(oc).astype(np.int32))
        if exact:
            assert not d.any() and np.array_equal(gs, os_), f"{name} {nm}: INT8 entries differ from the oracle's"
        if _active_rel[0] == REL_L2:
            allowed = np.ones(d.shape[:-1], np.int64)
        else:  # per head vector: the rounding step + the float bound in steps
            ov = np.asarray(oc, np.float64) * np.asarray(os_, np.float64)[..., None]
            nrm = np.linalg.norm(ov, axis=-1)
            mxv = np.max(np.abs(ov), axis=-1)
            allowed = 1 + np.ceil(127 * _active_rel[0] * nrm / np.where(mxv > 0, mxv, 1.0)).astype(np.int64)
            gv = gc.astype(np.float64) * gs.astype(np.float64)[..., None]
            stats.note(*check_close(f"{name} {nm} values", gv.reshape(-1, gv.shape[-1]), ov.reshape(-1, ov.shape[-1])))
        worst = d.max(axis=-1) - allowed
        assert worst.max(initial=-1) <= 0, f"{name} {nm}: a code differs by {d.max()} steps (allowed {allowed.max()})"
        stats.kv_codes += d.size
        stats.kv_code_steps += int(np.count_nonzero(d))
    stats.kv_checks += 1


def resync_rows(ctx, cfg, res, div, row_map):
    """Give the library the oracle's cache entries of this step for the layers
    above a near-tie divergence (the oracle's K/V are fp16 values already)."""
    for i, l in enumerate(div):
        r, s = row_map[i], int(res.slots[i])
        for m in range(l + 1, cfg.n_layers):
            if cfg.kv_int8:
                kc, ks, vc, vs = res.kv_entries[m][i]
                ctx.uocr_kv_write_i8(r, m, s, kc[:, None, :], ks[:, None], vc[:, None, :], vs[:, None])
                continue
            k = res.k_new[m, i].astype(np.float16)[:, None, :]
            v = res.v_new[m, i].astype(np.float16)[:, None, :]
            ctx.uocr_kv_write(r, m, s, k, v)


CHUNK = 64  # tokens of one prefill pass of the library


def library_prefill(ctx, wl, rows, row_map=(), moe_layers=()):
    """Build every row's prefix with uocr_prefill: the image embeddings, then
    the prompt ids (the workload's prefix).  Rows the oracle follows (row_map)
    are prefilled one 64-token call at a time (the library's own chunking) so
    that the router's choice for every prefix token can be read back from the
    debug taps after each call.  Returns the next id and the logits after each
    row's last prefix token, lib_sets[row][position][layer] = sorted experts
    the library chose (followed rows only), and the token count of the last
    call (its tokens are the ones the layer taps hold)."""
    import torch

    cfg = wl.cfg
    dev = torch.device("cuda")
    ne, P = wl.prefill_embeds.shape[1], cfg.prefix_len
    nxt = torch.zeros(rows, dtype=torch.int32, device=dev)
    lg = torch.zeros((rows, cfg.vocab), dtype=torch.float32, device=dev)
    lib_sets = {}
    for r in range(rows):
        x = torch.from_numpy(np.ascontiguousarray(wl.prefill_embeds[r]).view(np.int16)).to(dev)
        ids = torch.from_numpy(np.ascontiguousarray(wl.prefill_ids[r], np.int32)).to(dev)
        follow = r in row_map
        step = CHUNK if follow else P
        sets = {}
        for a in range(0, P, step):
            b = min(P, a + step)
            for lo, hi, kind in ((a, min(b, ne), "x"), (max(a, ne), b, "ids")):
                if lo >= hi:
                    continue
                last = hi == P
                n_last = hi - lo
                kw = dict(next_ptr=nxt[r:].data_ptr(), logits_ptr=lg[r].data_ptr()) if last else {}
                if kind == "x":
                    ctx.uocr_prefill(r, hi - lo, lo, x_ptr=x[lo:].data_ptr(), **kw)
                else:
                    ctx.uocr_prefill(r, hi - lo, lo, ids_ptr=ids[lo - ne:].data_ptr(), **kw)
                if follow:
                    for l in moe_layers:
                        idx = ctx.uocr_debug_router(l, hi - lo)["idx"]
                        for t in range(hi - lo):
                            sets.setdefault(lo + t, {})[l] = sorted(int(e) for e in idx[t])
        ctx.uocr_sync()
        lib_sets[r] = sets
    return nxt.cpu().numpy().copy(), lg.cpu().numpy().copy(), lib_sets, n_last


def compare_prefill(ctx, cfg, res, lib_rows, lib_next, lib_logits, stats, row_map, n_last_call, pk, pv, tie):
    """After the prefix: each layer's cached keys and values of the prefix, the
    layer taps of the last prefix token of the last prefilled row, and the
    logits / next id after each compared row's last prefix token.

    pk, pv: the oracle's prefix caches per layer [rows][nh][P][D]; tie[i][p]:
    the first MoE layer at which the library took another (equally correct,
    near-tie) expert set for row i at position p (n_layers if none).  From the
    layer after it that token's keys and values are not compared (the decode
    comparison's rule) and are replaced by the oracle's before decoding goes
    on."""
    P, L = cfg.prefix_len, cfg.n_layers
    for i, r in enumerate(row_map):
        for l in range(L):
            keep = [p for p in range(P) if tie[i][p] >= l]
            if cfg.kv_int8:  # the oracle's entries: its cached values are scale * code
                okc, oks = oracle_kv_quant(pk[l][i][:, keep])
                ovc, ovs = oracle_kv_quant(pv[l][i][:, keep])
                kc, ks, vc, vs = ctx.uocr_kv_read_i8(r, l, 0, P)
                check_int8_entries((kc[:, keep], ks[:, keep], vc[:, keep], vs[:, keep]), (okc, oks, ovc, ovs), stats,
                                   f"prefill row {r} layer {l}")
            else:
                k, v = ctx.uocr_kv_read(r, l, 0, P)
                stats.note(*check_close(f"prefill row {r} layer {l} keys", k[:, keep].astype(np.float64),
                                        pk[l][i][:, keep]))
                stats.note(*check_close(f"prefill row {r} layer {l} values", v[:, keep].astype(np.float64),
                                        pv[l][i][:, keep]))
                stats.kv_checks += 1
            for p in range(P):
                if tie[i][p] < l:  # the library's cache takes the oracle's entries
                    if cfg.kv_int8:
                        kq, vq = oracle_kv_quant(pk[l][i][:, p:p + 1]), oracle_kv_quant(pv[l][i][:, p:p + 1])
                        ctx.uocr_kv_write_i8(r, l, p, kq[0], kq[1], vq[0], vq[1])
                    else:
                        ctx.uocr_kv_write(r, l, p, pk[l][i][:, p:p + 1].astype(np.float16),
                                          pv[l][i][:, p:p + 1].astype(np.float16))
        stats.id_checks += 1
        if tie[i][P - 1] < L:
            stats.id_near_ties += 1
            continue
        stats.note(*check_close(f"prefill row {r} last-token logits", lib_logits[r], res.logits[i]))
        if res.margin[i] > ID_MARGIN:
            assert int(lib_next[r]) == int(res.next_ids[i]), f"prefill row {r}: id {lib_next[r]} != {res.next_ids[i]}"
        else:
            stats.id_near_ties += 1
    # the last uocr_prefill call (the prompt ids of the last row) left its
    # n_last_call tokens in the layer taps; its last token is position P - 1
    last = lib_rows - 1
    if last in row_map:
        i = row_map.index(last)
        n_tok = n_last_call
        t = tie[i][P - 1]
        for l in range(min(t + 1, L)):
            g = ctx.uocr_debug_hidden(2 * l, n_tok)[n_tok - 1:n_tok]
            stats.note(*check_close(f"prefill row {last} layer {l} after attention", g, res.h_attn[l][i:i + 1]))
            if l < t:
                g = ctx.uocr_debug_hidden(2 * l + 1, n_tok)[n_tok - 1:n_tok]
                stats.note(*check_close(f"prefill row {last} layer {l} output", g, res.hidden[l + 1][i:i + 1]))


def run_parity(ctx, wl, steps, oracle_model, **kw):
    """Run `steps` decode steps (plus the prefill-by-decode prefix when the
    workload has one) on both sides and compare.  With lib_prefill the library
    builds the prefix with uocr_prefill (one call per row and input kind)
    while the oracle takes its decode steps, and the two are compared once
    the prefix is complete.  Workloads with int8 activations take their own
    per-vector bound and must keep the median within the plain one.  Returns
    Stats."""
    a8 = bool(getattr(wl.cfg, "act_int8", 0))
    _active_rel[0] = REL_L2_INT8_ACT if a8 else REL_L2
    _active_abs[0] = MAX_ABS_INT8_ACT if a8 else MAX_ABS
    try:
        st = _run_parity(ctx, wl, steps, oracle_model, **kw)
    finally:
        _active_rel[0] = REL_L2
        _active_abs[0] = MAX_ABS
    if a8:
        med = float(np.median(st.rels))
        print(f"int8 activations: median rel-L2 {med:.2e}, 99th percentile {np.percentile(st.rels, 99):.2e}")
        assert med <= REL_L2, f"median rel-L2 {med:.3e} above {REL_L2} with int8 activations"
    return st


def _run_parity(ctx, wl, steps, oracle_model, rows=None, row_map=None, check_kv=True, log=None,
                same_router_input=False, lib_prefill=False):
    cfg = wl.cfg
    runner = LibraryRunner(ctx, wl, rows)
    n_or = oracle_model.rows
    row_map = list(range(n_or)) if row_map is None else row_map
    stats = Stats()
    plan = []
    last_ids = None if wl.first_ids is None else wl.first_ids.copy()
    if lib_prefill:
        assert wl.prefill_embeds is not None
        moe_layers = [l for l in range(cfg.n_layers) if not cfg.is_dense(l)]
        lib_next, lib_logits, lib_sets, n_last = library_prefill(ctx, wl, runner.rows, row_map, moe_layers)
        ne = wl.prefill_embeds.shape[1]
        res = None
        # tie[i][p]: first MoE layer at which the library's set for row i at position p
        # differs from the oracle's (only allowed where the oracle's gap is a near tie)
        tie = [[cfg.n_layers] * cfg.prefix_len for _ in range(n_or)]
        for p in range(cfg.prefix_len):
            opos = np.full(n_or, p, np.int32)
            last = p == cfg.prefix_len - 1
            if p < ne:
                res = oracle_model.step(opos, x=wl.prefill_embeds[row_map, p], want_logits=last)
            else:
                res = oracle_model.step(opos, ids=wl.prefill_ids[row_map, p - ne], want_logits=last)
            for i, r in enumerate(row_map):
                for l in moe_layers:
                    if tie[i][p] < cfg.n_layers:
                        break
                    want = sorted(int(e) for e in res.router[l]["idx"][i])
                    got = lib_sets[r][p][l]
                    stats.router_checks += 1
                    if got != want:
                        assert res.router[l]["gap"][i] <= ROUTER_GAP, \
                            f"prefill row {r} position {p} layer {l}: router set {got} != {want} with " \
                            f"oracle gap {res.router[l]['gap'][i]:.3e}"
                        stats.router_near_ties += 1
                        tie[i][p] = l
        compare_prefill(ctx, cfg, res, runner.rows, lib_next, lib_logits, stats, row_map, n_last,
                        oracle_model.pk, oracle_model.pv, tie)
        nxt = lib_next.copy()
        for i, r in enumerate(row_map):
            nxt[r] = res.next_ids[i]  # teacher forcing by the oracle
        last_ids = nxt
    elif wl.prefill_embeds is not None:
        ne = wl.prefill_embeds.shape[1]
        for p in range(cfg.prefix_len):
            if p < ne:
                plan.append(("x", p, wl.prefill_embeds[:, p]))
            else:
                plan.append(("ids", p, wl.prefill_ids[:, p - ne]))
    for s in range(steps):
        p = wl.start_pos + s
        if wl.step_x is not None:
            plan.append(("x", p, wl.step_x[s]))
        else:
            plan.append(("greedy", p, None))
    for si, (kind, p, data) in enumerate(plan):
        gpos = np.full(runner.rows, p, np.int32)
        opos = np.full(n_or, p, np.int32)
        is_last_prefill = wl.prefill_embeds is not None and p == cfg.prefix_len - 1
        want_lm = cfg.vocab > 0 and (kind == "greedy" or is_last_prefill)
        if kind == "x":
            g = runner.step(gpos, x=data[:runner.rows], want_logits=want_lm)
            res = oracle_model.step(opos, x=data[row_map], want_logits=want_lm)
        else:
            ids = data if kind == "ids" else last_ids
            g = runner.step(gpos, ids=ids[:runner.rows], want_logits=want_lm)
            res = oracle_model.step(opos, ids=ids[row_map], want_logits=want_lm)
        div = compare_step(ctx, cfg, res, runner.rows, stats, row_map=row_map, check_kv=check_kv,
                           same_router_input=same_router_input)
        resync_rows(ctx, cfg, res, div, row_map)
        clean = [i for i in range(n_or) if div[i] >= cfg.n_layers]
        if "y" in g and clean:
            stats.note(*check_close(f"step {si} output", g["y"][[row_map[i] for i in clean]],
                                    res.hidden[-1][clean]))
        if want_lm and clean:
            gl = g["logits"][[row_map[i] for i in clean]]
            stats.note(*check_close(f"step {si} logits", gl, res.logits[clean]))
            for i in clean:
                stats.id_checks += 1
                if res.margin[i] > ID_MARGIN:
                    assert int(g["next"][row_map[i]]) == int(res.next_ids[i]), \
                        f"step {si} row {row_map[i]}: argmax {g['next'][row_map[i]]} != {res.next_ids[i]}"
                else:
                    stats.id_near_ties += 1
        if want_lm:
            # teacher forcing: the oracle's greedy ids feed both sides (library rows outside
            # the oracle's sample keep their own argmax)
            nxt = g["next"].copy()
            for i, r in enumerate(row_map):
                nxt[r] = res.next_ids[i]
            last_ids = nxt
        stats.steps += 1
        stats.last_ids = last_ids  # the ids the next greedy step takes
        if log and (si % 50 == 0):
            log(f"step {si}/{len(plan)} worst rel {stats.worst_rel:.2e}")
    return stats
