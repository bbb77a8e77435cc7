"""Free-running parity of the CUDA library (through the C ABI) against the oracle.

Both sides consume the same seeded workload; nothing the library computes is
ever an input of the oracle.  For token-id workloads the library is fed the
oracle's greedy ids (teacher forcing by the oracle), so a near-tie argmax
cannot make the two inputs diverge.

Comparison rules (the decode-step statement's tolerances):
* every floating-point output (hidden state after attention and after each
  layer, the K and V written to the cache, LM logits): relative L2 error
  <= 2e-3 and max abs error <= 2e-2 against the oracle;
* integer outputs bit-exact: the router's top-k set where the oracle's k-th
  vs (k+1)-th logit gap exceeds 1e-2, argmax ids where the oracle's top-2
  margin exceeds 1e-2, the counts / offsets / permutation of the grouping
  (equal to the oracle's when every row's set matches, else checked to be
  the stable grouping of the library's own top-k); the library's set is
  always exactly the top-k of its own fp32 logits;
* router logits and routing weights are intermediates: logits to max-abs
  5e-3 per unit of logit magnitude, weights to rel-L2 1e-2; the layer output
  they feed keeps the full tolerance; router sets are compared wherever the
  oracle's gap exceeds both 1e-2 and twice the observed logit difference,
  which makes the comparison sound;
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
MAX_ABS = 2e-2
ROUTER_GAP = oracle.TIE_TOL  # router sets are compared where the oracle's gap exceeds it
ID_MARGIN = 1e-2
WEIGHTS_REL = 1e-2  # routing weights: an intermediate (see compare_step)
ROUTER_LOGIT_REL = 5e-3  # router logits: an intermediate, max-abs error per unit of logit magnitude


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def check_close(name, got, want, rel=REL_L2, mx=MAX_ABS):
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
    tainted_rows: set = field(default_factory=set)

    worst_name: str = ""

    def note(self, e, m, name=""):
        self.float_checks += 1
        if e > self.worst_rel:
            self.worst_name = name
        self.worst_rel = max(self.worst_rel, e)
        self.worst_abs = max(self.worst_abs, m)


class GpuRunner:
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


def compare_step(ctx, cfg, res, lib_rows, stats, row_map=None, check_kv=True):
    """Compare one step.  res: oracle StepResult over the oracle's rows;
    row_map[i] = library row of oracle row i.  Returns, per oracle row, the
    layer whose MoE output diverged at a router near tie (cfg.n_layers if none)."""
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
                # The library's logits stay within a small multiple of their magnitude of
                # the oracle's; the sets must then agree wherever the oracle's k-th vs
                # (k+1)-th gap exceeds twice the observed difference (and the 1e-2 gate).
                err = float(np.max(np.abs(glog[r].astype(np.float64) - info["logits"][i])))
                scale = max(1.0, float(np.max(np.abs(info["logits"][i]))))
                assert err <= ROUTER_LOGIT_REL * scale, \
                    f"layer {l} row {r}: router logits differ by {err:.3e} (scale {scale:.2f})"
                gate = max(ROUTER_GAP, 2 * err)
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
                stats.note(*check_close(f"layer {l} row {r} routing weights", got_w, info["w"][i],
                                        rel=WEIGHTS_REL))
            # grouping: unique given the top-k sets
            flat = gr["idx"].reshape(-1)
            E = cfg.n_experts
            assert np.array_equal(gr["count"], np.bincount(flat, minlength=E)), f"layer {l}: counts"
            assert np.array_equal(gr["offset"], np.concatenate([[0], np.cumsum(gr["count"])])), f"layer {l}: offsets"
            assert np.array_equal(gr["perm"], np.argsort(flat, kind="stable")), f"layer {l}: permutation"
            if router_all_equal and n == lib_rows and row_map == list(range(n)):
                # unique part of the grouping: the (row, expert) sequence; the slot
                # numbers inside a row depend on the order of near-equal chosen logits
                k = cfg.top_k
                assert np.array_equal(gr["count"], info["count"]), f"layer {l}: counts vs oracle"
                assert np.array_equal(gr["offset"], info["offset"]), f"layer {l}: offsets vs oracle"
                g_pairs = [(int(e) // k, int(gr["idx"][e // k][e % k])) for e in gr["perm"]]
                o_pairs = [(int(e) // k, int(info["idx"][e // k][e % k])) for e in info["perm"]]
                assert g_pairs == o_pairs, f"layer {l}: grouping {g_pairs} != {o_pairs}"

        if out_ok:
            g = tap(2 * l + 1)[[row_map[i] for i in out_ok]]
            stats.note(*check_close(f"layer {l} output", g, res.hidden[l + 1][out_ok]))
    return div


def resync_rows(ctx, cfg, res, div, row_map):
    """Give the library the oracle's cache entries of this step for the layers
    above a near-tie divergence (the oracle's K/V are fp16 values already)."""
    for i, l in enumerate(div):
        r, s = row_map[i], int(res.slots[i])
        for m in range(l + 1, cfg.n_layers):
            k = res.k_new[m, i].astype(np.float16)[:, None, :]
            v = res.v_new[m, i].astype(np.float16)[:, None, :]
            ctx.uocr_kv_write(r, m, s, k, v)


def run_parity(ctx, wl, steps, oracle_model, rows=None, row_map=None, check_kv=True, log=None):
    """Run `steps` decode steps (plus the prefill-by-decode prefix when the
    workload has one) on both sides and compare.  Returns Stats."""
    cfg = wl.cfg
    runner = GpuRunner(ctx, wl, rows)
    n_or = oracle_model.rows
    row_map = list(range(n_or)) if row_map is None else row_map
    stats = Stats()
    plan = []
    if wl.prefill_embeds is not None:
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
    last_ids = None if wl.first_ids is None else wl.first_ids.copy()
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
        div = compare_step(ctx, cfg, res, runner.rows, stats, row_map=row_map, check_kv=check_kv)
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
