"""Pins of the float64 oracle against things other than itself.

Each test ties one oracle part to a closed form, an invariant, a library
routine, a hand-built fixture, or the independent scalar statement in
tests/bruteforce.py, chosen so that a dropped term, a wrong sign or index or a
transposed operand fails at least one of them.
"""
import math
import os

import numpy as np
import pytest

import oracle
from oracle import model as om
from oracle.quant import dequant, float32_is_exact
from quantized_moe_decode_gb300 import synth

from bruteforce import BruteModel, decode_rows, rot

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
FMT = {"q8_0": 1, "q4_0": 2, "i8asym": 3, "q8_0_g64": 4, "q4_0_g64": 5}


# ------------------------------------------------------------------ dequantisation
def _golden_blocks():
    out = []
    with open(os.path.join(GOLDEN, "quant_blocks.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            left, right = line.split("|")
            name, hexs = left.split()
            out.append((name, bytes.fromhex(hexs), [float(v) for v in right.split()]))
    return out


@pytest.mark.parametrize("case", range(11))
def test_hand_built_blocks_dequantise_exactly(case):
    name, raw, expected = _golden_blocks()[case]
    got = dequant(np.frombuffer(raw, np.uint8), FMT[name], 1, len(expected))[0]
    assert got.tolist() == expected


@pytest.mark.parametrize("fmt", [synth.F16, synth.Q8_0, synth.Q4_0, synth.I8ASYM, synth.Q8_0_G64, synth.Q4_0_G64])
def test_dequant_matches_scalar_parser(fmt):
    rng = np.random.default_rng(7)
    x = rng.standard_normal((5, 128), dtype=np.float32) * 0.02
    t = synth.Tensor(0, 0, 0, fmt, 5, 128, synth.encode(x, fmt))
    got = dequant(t.blob, fmt, 5, 128)
    ref = np.array(decode_rows(t))
    assert np.array_equal(got, ref)
    # and the encoding is a faithful quantisation of the draw (catches a wrong scale / sign)
    assert np.max(np.abs(got - x)) < (0.02 * 4 / 7 if fmt in (synth.Q4_0, synth.Q4_0_G64) else 0.02 * 4 / 100)


def test_q8_q4_values_are_exact_in_float32():
    rng = np.random.default_rng(8)
    for fmt in (synth.Q8_0, synth.Q4_0, synth.I8ASYM, synth.Q8_0_G64, synth.Q4_0_G64):
        x = rng.standard_normal((7, 128), dtype=np.float32)
        w = dequant(synth.encode(x, fmt), fmt, 7, 128)
        assert float32_is_exact(w)


# ------------------------------------------------------------------ elementwise parts
def test_rmsnorm_unit_rms_and_scale_invariance():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(1280) * 3.7
    y = om.rmsnorm(x, np.ones(1280), 0.0)
    assert abs(math.sqrt(np.mean(y * y)) - 1.0) < 1e-12
    assert np.allclose(om.rmsnorm(5.0 * x, np.ones(1280), 0.0), y, rtol=1e-12, atol=0)
    w = rng.standard_normal(1280)
    assert np.allclose(om.rmsnorm(x, w, 0.0), y * w, rtol=1e-12, atol=0)
    # eps enters inside the root: a zero vector stays zero, a tiny one is damped
    assert np.all(om.rmsnorm(np.zeros(8), np.ones(8), 1e-6) == 0)
    t = np.full(4, 1e-3)
    assert np.allclose(om.rmsnorm(t, np.ones(4), 1e-6), t / math.sqrt(1e-6 + 1e-6))


def test_silu_closed_forms():
    assert om.silu(np.float64(0.0)) == 0.0
    z = np.linspace(-6, 6, 25)
    assert np.allclose(om.silu(z) - om.silu(-z), z, atol=1e-14)
    assert np.allclose(om.silu(z), z / (1 + np.exp(-z)))
    assert abs(om.silu(np.float64(40.0)) - 40.0) < 1e-12


def test_rope_identity_norm_and_relative_position():
    rng = np.random.default_rng(2)
    q = rng.standard_normal(128)
    k = rng.standard_normal(128)
    assert np.array_equal(om.rope(q, 0, 1e4), q)
    for p in (1, 17, 300, 3000):
        assert abs(np.linalg.norm(om.rope(q, p, 1e4)) - np.linalg.norm(q)) < 1e-12
    # <R_p q, R_p' k> depends only on p - p'
    a = om.rope(q, 310, 1e4) @ om.rope(k, 300, 1e4)
    b = om.rope(q, 10, 1e4) @ om.rope(k, 0, 1e4)
    assert abs(a - b) < 1e-10


def test_rope_pairs_first_and_second_half_like_complex_rotation():
    # D = 2: a plain rotation by angle p
    v = np.array([0.3, -1.2])
    p = 5
    c, s = math.cos(p), math.sin(p)
    assert np.allclose(om.rope(v, p, 1e4), [0.3 * c + 1.2 * s, -1.2 * c + 0.3 * s])
    # D = 16: pair (i, i + 8) rotates as the complex number v[i] + 1j*v[i+8]
    rng = np.random.default_rng(3)
    v = rng.standard_normal(16)
    assert np.allclose(om.rope(v, 37, 1e4), rot(list(v), 37, 1e4), atol=1e-13)


def test_ring_slot_closed_cases():
    assert [om.ring_slot(p, 289, 128) for p in (0, 288, 289, 416, 417, 418, 588)] == \
        [0, 288, 289, 416, 289, 290, 289 + (588 - 289) % 128]


# ------------------------------------------------------------------ attention
def test_attention_single_key_and_equal_logits():
    rng = np.random.default_rng(4)
    q = rng.standard_normal(64)
    K = rng.standard_normal((1, 64))
    V = rng.standard_normal((1, 64))
    assert np.allclose(om.attend(q, K, V), V[0])
    K = np.zeros((5, 64))
    V = rng.standard_normal((5, 64))
    assert np.allclose(om.attend(q, K, V), V.mean(axis=0))


def test_attention_two_keys_closed_form_and_scale():
    q = np.zeros(4)
    q[0] = 2.0
    K = np.array([[1.0, 0, 0, 0], [0.0, 0, 0, 0]])
    V = np.array([[1.0, 0, 0, 0], [0.0, 1, 0, 0]])
    # logits 2*1/sqrt(4) = 1 and 0 -> weights sigmoid(1), sigmoid(-1)
    s1 = 1 / (1 + math.exp(-1.0))
    assert np.allclose(om.attend(q, K, V), [s1, 1 - s1, 0, 0])


def test_attention_split_merge_equals_one_pass():
    rng = np.random.default_rng(5)
    q, K, V = rng.standard_normal(128), rng.standard_normal((300, 128)), rng.standard_normal((300, 128))
    o, lse = om.attend_lse(q, K, V)
    parts = [om.attend_lse(q, K[a:b], V[a:b]) for a, b in ((0, 77), (77, 200), (200, 300))]
    M = max(l for _, l in parts)
    w = np.array([math.exp(l - M) for _, l in parts])
    merged = sum(wi * oi for wi, (oi, _) in zip(w, parts)) / w.sum()
    assert np.allclose(merged, o, atol=1e-12)
    assert abs(M + math.log(w.sum()) - lse) < 1e-12


def test_sink_key_equals_sigmoid_rescale():
    """Falcon-OCR card: output * sigmoid(lse - sink) == softmax with one more zero-value key."""
    rng = np.random.default_rng(6)
    for s in (-3.0, 0.0, 0.7, 5.0):
        q, K, V = rng.standard_normal(64), rng.standard_normal((40, 64)), rng.standard_normal((40, 64))
        o, lse = om.attend_lse(q, K, V)
        assert np.allclose(om.attend(q, K, V, sink=s), o / (1 + math.exp(-(lse - s))), atol=1e-13)
    assert np.allclose(om.attend(q, K, V, sink=-1e4), o, atol=1e-13)


# ------------------------------------------------------------------ routing
def test_route_selection_weights_and_ties():
    lg = np.array([0.1, 2.0, -1.0, 2.0, 0.5, 2.0])
    idx, w = om.route(lg, 2)
    assert idx.tolist() == [1, 3]             # lowest indices among the tied maxima
    assert np.allclose(w, [0.5, 0.5])
    idx, w = om.route(lg, 1)
    assert idx.tolist() == [int(np.argmax(lg))] and w.tolist() == [1.0]
    rng = np.random.default_rng(9)
    lg = rng.standard_normal(64)
    idx, w = om.route(lg, 6)
    assert abs(w.sum() - 1) < 1e-14
    assert set(idx.tolist()) == set(np.argsort(lg)[-6:].tolist())
    # ratio of two weights is exp of the logit difference
    assert abs(w[0] / w[1] - math.exp(lg[idx[0]] - lg[idx[1]])) < 1e-12
    # k = E: the renormalised weights are the full softmax
    idx, w = om.route(lg, 64)
    sm = np.exp(lg - lg.max()) / np.exp(lg - lg.max()).sum()
    assert np.allclose(w, sm[idx], atol=1e-15)


def test_grouping_is_a_stable_sort_by_expert():
    rng = np.random.default_rng(10)
    for rows, k, E in ((1, 6, 64), (8, 6, 64), (64, 6, 64), (5, 2, 4)):
        idx = np.stack([rng.permutation(E)[:k] for _ in range(rows)])
        count, offset, perm = om.group_by_expert(idx, E)
        assert np.array_equal(count, np.bincount(idx.reshape(-1), minlength=E))
        assert np.array_equal(offset, np.concatenate([[0], np.cumsum(count)]))
        assert np.array_equal(perm, np.argsort(idx.reshape(-1), kind="stable"))


def _tiny_cfg(**kw):
    base = dict(hidden=32, n_heads=2, head_dim=16, n_layers=3, n_dense_layers=1, dense_inter=64,
                n_experts=4, top_k=2, n_shared=2, expert_inter=32, vocab=10, fmt_attn=synth.Q8_0,
                fmt_dense=synth.Q8_0, fmt_shared=synth.Q8_0, fmt_routed=synth.Q4_0,
                prefix_len=3, ring_len=4, max_rows=2)
    base.update(kw)
    return synth.ModelConfig(**base)


def test_top_all_experts_equals_dense_softmax_mixture():
    cfg = _tiny_cfg(n_layers=1, n_dense_layers=0, top_k=4, n_shared=0, vocab=0)
    wl = synth.make_workload("t", cfg, 2, 1, 11)
    m = oracle.OracleModel(cfg, wl.tensors, 2, kv_prefix=wl.kv_prefix)
    res = m.step(wl.positions(0), x=wl.step_x[0])
    Hh = res.h_attn[0]
    # the method stores the normalised input and the SwiGLU activations in fp16
    Hn = om.rmsnorm(Hh, m.w(om.T_MLP_NORM, 0), cfg.rms_eps).astype(np.float16).astype(np.float64)

    def expert(x, e):
        g, u = m.w(om.T_EXPERT_GATE, 0, e) @ x, m.w(om.T_EXPERT_UP, 0, e) @ x
        a = (g / (1 + np.exp(-g)) * u).astype(np.float16).astype(np.float64)
        return m.w(om.T_EXPERT_DOWN, 0, e) @ a

    for r in range(2):
        lg = m.w(om.T_ROUTER, 0) @ Hn[r]
        p = np.exp(lg - lg.max())
        p /= p.sum()
        mix = sum(p[e] * expert(Hn[r], e) for e in range(4))
        assert np.allclose(res.hidden[1][r], Hh[r] + mix, atol=1e-12)


def test_two_shared_experts_equal_one_concatenated_expert():
    rng = np.random.default_rng(12)
    x = rng.standard_normal(32)
    g = [rng.standard_normal((16, 32)) for _ in range(2)]
    u = [rng.standard_normal((16, 32)) for _ in range(2)]
    d = [rng.standard_normal((32, 16)) for _ in range(2)]
    two = om.swiglu(x, g[0], u[0], d[0]) + om.swiglu(x, g[1], u[1], d[1])
    one = om.swiglu(x, np.vstack(g), np.vstack(u), np.hstack(d))
    assert np.allclose(two, one, atol=1e-12)


def test_fp16_storage_rounds_to_nearest_even():
    u = 2.0 ** -10  # fp16 spacing at 1
    assert om.f16(1 + u / 2) == 1.0                  # tie -> even mantissa
    assert om.f16(1 + 3 * u / 2) == 1 + 2 * u        # tie -> even mantissa (up)
    assert om.f16(1 + 0.51 * u) == 1 + u
    with np.errstate(over="ignore"):
        assert om.f16(65504.0) == 65504.0 and np.isinf(om.f16(65520.0))
    assert om.f16(-2.0 ** -24) == -2.0 ** -24        # smallest subnormal survives
    x = np.random.default_rng(13).standard_normal(1000)
    assert np.all(np.abs(om.f16(x) - x) <= np.abs(x) * 2.0 ** -11 + 2.0 ** -25)


def test_argmax_first_maximum():
    assert om.argmax_first(np.array([1.0, 3.0, 3.0, -1.0])) == 1
    assert om.argmax_first(np.array([-2.0])) == 0


# ------------------------------------------------------------------ whole step vs brute force
def _compare_with_brute(cfg, rows, steps, seed, prefix="cached", n_embeds=0, ids=False):
    wl = synth.make_workload("t", cfg, rows, steps, seed, prefix=prefix,
                             n_prefill_embeds=n_embeds, step_input="ids" if ids else "x")
    orc = oracle.OracleModel(cfg, wl.tensors, rows, kv_prefix=wl.kv_prefix, sinks=wl.sinks)
    bru = BruteModel(cfg, wl.tensors, rows, kv_prefix=wl.kv_prefix, sinks=wl.sinks)
    plan = []
    if prefix == "prefill":
        for p in range(cfg.prefix_len):
            pos = np.full(rows, p, np.int32)
            if p < n_embeds:
                plan.append((pos, None, wl.prefill_embeds[:, p]))
            else:
                plan.append((pos, wl.prefill_ids[:, p - n_embeds], None))
    for s in range(steps):
        pos = wl.positions(s)
        if ids:
            plan.append((pos, "greedy", None))
        else:
            plan.append((pos, None, wl.step_x[s]))
    last = None
    for pos, idv, x in plan:
        if isinstance(idv, str):
            idv = last.next_ids if last is not None and last.next_ids is not None else wl.first_ids
        a = orc.step(pos, ids=idv, x=x)
        b = bru.step(pos, ids=idv, x=x)
        for r in range(rows):
            layers, logits = b[r]
            for l in range(cfg.n_layers):
                assert np.allclose(a.hidden[l + 1][r], layers[l], rtol=1e-10, atol=1e-10), (pos, l, r)
            if logits is not None:
                assert np.allclose(a.logits[r], logits, rtol=1e-10, atol=1e-10)
        last = a
    return orc


def test_tiny_moe_model_matches_brute_force_through_ring_wrap():
    # prefix of 3 built by decode (2 embeddings + 1 token), then 7 greedy steps, ring of 4
    _compare_with_brute(_tiny_cfg(), rows=2, steps=7, seed=13, prefix="prefill", n_embeds=2, ids=True)


def test_tiny_dense_sink_model_matches_brute_force():
    cfg = _tiny_cfg(n_layers=2, n_dense_layers=2, n_experts=0, top_k=0, n_shared=0, vocab=0,
                    fmt_attn=synth.I8ASYM, fmt_dense=synth.I8ASYM, use_sink=1, prefix_len=5)
    _compare_with_brute(cfg, rows=2, steps=6, seed=14)


def test_tiny_q4_attention_cached_prefix_matches_brute_force():
    cfg = _tiny_cfg(n_layers=2, n_dense_layers=1, fmt_attn=synth.Q4_0, fmt_shared=synth.Q4_0, vocab=0,
                    prefix_len=6, ring_len=3)
    _compare_with_brute(cfg, rows=1, steps=5, seed=15)


def test_ring_equals_full_attention_while_generated_fits():
    """With g <= R the ring holds every generated token: same as an unbounded cache."""
    cfg = _tiny_cfg(n_layers=2, n_dense_layers=1, vocab=0, ring_len=6)
    big = cfg.replace(ring_len=1000)
    wl = synth.make_workload("t", cfg, 2, 6, 16)
    a = oracle.OracleModel(cfg, wl.tensors, 2, kv_prefix=wl.kv_prefix)
    b = oracle.OracleModel(big, wl.tensors, 2, kv_prefix=wl.kv_prefix)
    for s in range(6):
        ra = a.step(wl.positions(s), x=wl.step_x[s])
        rb = b.step(wl.positions(s), x=wl.step_x[s])
        assert np.array_equal(ra.hidden, rb.hidden)
    # one step more and the oldest generated token has left the ring
    x = wl.step_x[0]
    ra = a.step(wl.positions(6), x=x)
    rb = b.step(wl.positions(6), x=x)
    assert not np.allclose(ra.hidden[-1], rb.hidden[-1])


def test_float32_cache_gives_identical_results():
    cfg = _tiny_cfg(vocab=10)
    wl = synth.make_workload("t", cfg, 2, 2, 17, step_input="ids")
    a = oracle.OracleModel(cfg, wl.tensors, 2, kv_prefix=wl.kv_prefix, cache="float64")
    b = oracle.OracleModel(cfg, wl.tensors, 2, kv_prefix=wl.kv_prefix, cache="float32")
    ra = a.step(wl.positions(0), ids=wl.first_ids)
    rb = b.step(wl.positions(0), ids=wl.first_ids)
    assert np.array_equal(ra.logits, rb.logits)


# ---------------------------------------------------------------- INT8 KV cache
def test_kv_quant_hand_built_codes_and_scale():
    """amax 127 gives s = 1 exactly; codes round half to even; the amax maps to 127."""
    x = np.array([127.0, -63.5, 0.5, 1.5, 2.5, -2.5, 0.0, 126.5, -0.49])
    codes, s = oracle.kv_quant(x)
    assert s.dtype == np.float32 and float(s) == 1.0
    assert codes.tolist() == [127, -64, 0, 2, 2, -2, 0, 126, 0]
    # a power-of-two rescale changes the scale exactly and no code
    c2, s2 = oracle.kv_quant(x * 2.0 ** -9)
    assert float(s2) == 2.0 ** -9 and np.array_equal(c2, codes)
    assert np.array_equal(oracle.kv_dequant(codes, s), codes.astype(np.float64))


def test_kv_quant_negative_amax_zero_vector_and_shapes():
    codes, s = oracle.kv_quant(np.array([-3.0, 1.0, 0.25]))
    assert codes[0] == -127 and float(s) == np.float32(3.0) / np.float32(127.0)
    codes, s = oracle.kv_quant(np.zeros((2, 4)))
    assert not codes.any() and not s.any()
    codes, s = oracle.kv_quant(np.ones((3, 5, 8)))
    assert codes.shape == (3, 5, 8) and s.shape == (3, 5) and (codes == 127).all()


def test_kv_quant_round_trip_error_bound_and_code_range():
    rng = np.random.default_rng(7)
    x = rng.standard_normal((64, 128)) * rng.uniform(0.01, 10.0, size=(64, 1))
    codes, s = oracle.kv_quant(x)
    err = np.abs(oracle.kv_dequant(codes, s) - x)
    # half a step, plus the fp32 rounding of x / s
    assert (err <= s[:, None].astype(np.float64) * (0.5 + 1e-5) + 1e-7 * np.abs(x)).all()
    assert (np.abs(codes).max(axis=1) == 127).all() and np.abs(codes.astype(int)).max() <= 127


def test_int8_kv_model_caches_the_quantised_prefix_and_stays_close_to_fp16():
    cfg = synth.ModelConfig(hidden=128, n_heads=2, head_dim=64, n_layers=2, n_dense_layers=2, dense_inter=256,
                            prefix_len=10, ring_len=4, max_rows=2)
    wl = synth.make_workload("kvq", cfg, 2, 6, 11)
    kv = wl.kv_prefix.subset([0, 1])
    m8 = oracle.OracleModel(cfg, wl.tensors, 2, kv_prefix=kv, kv_int8=True)
    m16 = oracle.OracleModel(cfg, wl.tensors, 2, kv_prefix=kv)
    for l in range(cfg.n_layers):
        k, v = kv[l]
        assert np.array_equal(m8.pk[l], oracle.kv_dequant(*oracle.kv_quant(k)))
        assert np.array_equal(m8.pv[l], oracle.kv_dequant(*oracle.kv_quant(v)))
    for s in range(wl.steps):  # past the ring's wrap
        pos = np.full(2, cfg.prefix_len + s)
        r8 = m8.step(pos, x=wl.step_x[s])
        r16 = m16.step(pos, x=wl.step_x[s])
        # the appended entries are the quantised keys / values of this step
        for l in range(cfg.n_layers):
            c, sc = oracle.kv_quant(r8.k_new[l])
            assert np.array_equal(oracle.kv_dequant(c, sc), r8.k_new[l])
        d = np.linalg.norm(r8.hidden[-1] - r16.hidden[-1]) / np.linalg.norm(r16.hidden[-1])
        assert 0 < d < 2e-2, d  # int8 noise, not a different model


# ---------------------------------------------------------------- projector
def _q8_block_row(d_bits, codes):
    """One Q8_0 row from hand-built blocks: fp16 scale bits + 32 int8 codes per block."""
    out = bytearray()
    for i in range(0, len(codes), 32):
        out += int(d_bits).to_bytes(2, "little") + bytes((c + 256) % 256 for c in codes[i:i + 32])
    return out


def test_projector_one_hot_feature_selects_a_column_plus_bias():
    # W [4][64] from Q8_0 blocks with d = 2^-7 (fp16 0x2000) and codes W[r][k] = (r * 7 + k) % 21 - 10;
    # every value is k/128 exactly, so a one-hot feature gives column j plus the bias exactly in fp16
    rows, cols = 4, 64
    codes = [[(r * 7 + k) % 21 - 10 for k in range(cols)] for r in range(rows)]
    blob = np.frombuffer(b"".join(bytes(_q8_block_row(0x2000, codes[r])) for r in range(rows)), np.uint8)
    W = dequant(blob, synth.Q8_0, rows, cols)
    assert W[1, 3] == ((1 * 7 + 3) % 21 - 10) / 128.0
    b = np.array([0.5, -0.25, 0.0, 1.0])
    for j in (0, 13, 63):
        x = np.zeros((1, cols))
        x[0, j] = 2.0
        y = oracle.project(x, W, b)
        assert y[0].tolist() == [2.0 * codes[r][j] / 128.0 + b[r] for r in range(rows)]
    # without a bias the map is linear: opposite features give opposite outputs exactly
    x = np.zeros((2, cols))
    x[0, 5], x[1, 5] = 1.0, -1.0
    y = oracle.project(x, W)
    assert np.array_equal(y[0], -y[1])


def test_projector_output_is_fp16_of_the_exact_product():
    rng = np.random.default_rng(12)
    W = dequant(synth.encode(rng.standard_normal((8, 128), dtype=np.float32) * 0.02, synth.Q4_0_G64),
                synth.Q4_0_G64, 8, 128)
    x = rng.standard_normal((3, 128)).astype(np.float16).astype(np.float64)
    b = rng.standard_normal(8).astype(np.float16).astype(np.float64)
    y = oracle.project(x, W, b)
    exact = np.array([[sum(x[t, k] * W[r, k] for k in range(128)) + b[r] for r in range(8)] for t in range(3)])
    assert np.array_equal(y, exact.astype(np.float16).astype(np.float64))


# ---------------------------------------------------------------- dynamic int8 activations
def test_act_quant_groups_of_32_hand_built():
    # group 0: amax 127 -> s = 1, codes round half to even; group 1: all zero; group 2: s = 2^-3
    x = np.zeros(96)
    x[:32] = np.linspace(-127, 127, 32)
    x[5] = 2.5
    x[64:96] = np.arange(32) * 0.125 - 2.0
    y = oracle.act_quant(x)
    assert np.array_equal(y[:32][[0, 31]], [-127.0, 127.0]) and y[5] == 2.0
    assert not y[32:64].any()
    # group 2: amax 2.0 -> s = 2/127 (fp32); every value within half a step
    s2 = np.float32(2.0) / np.float32(127.0)
    assert np.all(np.abs(y[64:96] - x[64:96]) <= float(s2) / 2 + 1e-12)
    # per-group scale: multiplying one group by 2^k scales only that group's result
    x2 = x.copy()
    x2[64:96] *= 8.0
    y2 = oracle.act_quant(x2)
    assert np.array_equal(y2[64:96], 8.0 * y[64:96]) and np.array_equal(y2[:64], y[:64])


def test_int8_activation_grid_error_behind_the_parity_bound():
    # The int8-activation parity bound reads "every code one step apart" as about
    # sqrt(12) x the grid's own relative error eps_q; on N(0, 1) activations in
    # groups of 32 eps_q is 0.5-0.7% (group max / rms ~ 2.1-2.6), so the bound
    # sqrt(12) eps_q stays within 2.5e-2, and one step on every code is exactly
    # s per input, sqrt(12) times the uniform rounding error's rms.
    rng = np.random.default_rng(5)
    x = rng.standard_normal((4096, 32 * 32))
    q = oracle.act_quant(x)
    eps_q = np.linalg.norm(q - x) / np.linalg.norm(x)
    assert 0.004 < eps_q < 0.008, eps_q
    assert np.sqrt(12.0) * eps_q < 2.5e-2
    g = x.reshape(-1, 32)
    s = np.max(np.abs(g), axis=1) / 127.0
    step_err = np.sqrt(np.mean(s ** 2)) * np.sqrt(g.size / g.shape[0]) / np.sqrt(np.mean(np.sum(g ** 2, axis=1)))
    assert abs(step_err / eps_q - np.sqrt(12.0)) < 0.1 * np.sqrt(12.0)


def test_int8_activation_model_is_close_to_fp16_and_exact_on_its_grid():
    cfg = synth.ModelConfig(hidden=128, n_heads=2, head_dim=64, n_layers=2, n_dense_layers=2, dense_inter=256,
                            prefix_len=6, ring_len=4, max_rows=2)
    wl = synth.make_workload("actq", cfg, 2, 3, 13)
    kv = wl.kv_prefix.subset([0, 1])
    m8 = oracle.OracleModel(cfg, wl.tensors, 2, kv_prefix=kv, act_int8=True)
    m16 = oracle.OracleModel(cfg, wl.tensors, 2, kv_prefix=kv)
    for s in range(wl.steps):
        pos = np.full(2, cfg.prefix_len + s)
        r8 = m8.step(pos, x=wl.step_x[s])
        r16 = m16.step(pos, x=wl.step_x[s])
        d = np.linalg.norm(r8.hidden[-1] - r16.hidden[-1]) / np.linalg.norm(r16.hidden[-1])
        assert 0 < d < 3e-2, d
    # a vector already on the grid (codes times a power-of-two scale) is its own quantisation
    g = np.arange(-16, 16) * 2.0 ** -4
    g[0] = -127 * 2.0 ** -4
    assert np.array_equal(oracle.act_quant(g), g)
