"""GPU parity of the decode step against the float64 oracle on small models.

Sizes are chosen so the oracle finishes in seconds while every kernel still
spans several tiles and a ragged tail: rows that are not a multiple of the
8-token n-tile, several token groups (40 rows), a vocabulary that is not a
multiple of the 16-row slab (1000), ring wrap-around (ring of 8 slots), split
attention with empty splits, every weight format and every (routed, shared)
expert format pair the library supports.
"""
import numpy as np
import pytest

from quantized_moe_decode_gb300 import synth

from helpers import make_ctx, make_oracle
from parity import run_parity

pytestmark = pytest.mark.gpu

Q8, Q4, I8 = synth.Q8_0, synth.Q4_0, synth.I8ASYM


def _dense(**kw):
    base = dict(hidden=256, n_heads=4, head_dim=64, n_layers=2, n_dense_layers=2, dense_inter=512,
                fmt_attn=Q8, fmt_dense=Q8, prefix_len=20, ring_len=8, max_rows=3)
    base.update(kw)
    return synth.ModelConfig(**base)


def _moe(**kw):
    base = dict(hidden=256, n_heads=2, head_dim=128, n_layers=3, n_dense_layers=1, dense_inter=512,
                n_experts=16, top_k=4, n_shared=2, expert_inter=128, vocab=1000, fmt_attn=Q8, fmt_dense=Q8,
                fmt_shared=Q8, fmt_routed=Q4, prefix_len=12, ring_len=8, max_rows=5)
    base.update(kw)
    return synth.ModelConfig(**base)


def _run(wl, steps, **kw):
    ctx = make_ctx(wl)
    orc = make_oracle(wl)
    st = run_parity(ctx, wl, steps, orc, **kw)
    print(f"\n{wl.name}: {st.steps} steps, {st.float_checks} float checks (worst rel-L2 {st.worst_rel:.2e}, "
          f"max-abs {st.worst_abs:.2e}), router {st.router_checks} ({st.router_near_ties} near ties), "
          f"ids {st.id_checks} ({st.id_near_ties} near ties), kv {st.kv_checks}; worst: {st.worst_name}")
    ctx.close()
    return st


def test_dense_q8_ring_wrap(cuda):
    wl = synth.make_workload("dense_q8", _dense(), 3, 20, 100)
    st = _run(wl, 20)
    assert st.kv_checks == 20 * 2 * 3


def test_dense_q4_attention_i8asym_mlp_with_sinks(cuda):
    cfg = _dense(fmt_attn=Q4, fmt_dense=I8, use_sink=1, head_dim=32, n_heads=8, prefix_len=5)
    wl = synth.make_workload("dense_q4_i8_sink", cfg, 3, 12, 101)
    _run(wl, 12)


def test_dense_i8asym_sink_head_dim_64_single_row(cuda):
    cfg = _dense(fmt_attn=I8, fmt_dense=I8, use_sink=1, prefix_len=33, max_rows=1, hidden=128,
                 n_heads=2, dense_inter=256)
    wl = synth.make_workload("dense_i8_sink", cfg, 1, 12, 102)
    _run(wl, 12)


def test_moe_prefill_by_decode_then_greedy_with_lm_head(cuda):
    wl = synth.make_workload("moe_lm", _moe(), 5, 12, 103, prefix="prefill", n_prefill_embeds=8,
                             step_input="ids")
    st = _run(wl, 12)
    assert st.id_checks >= 5 * 12
    assert st.router_checks > 0


def test_moe_forty_rows_three_token_groups(cuda):
    cfg = _moe(max_rows=40, fmt_shared=Q4, fmt_routed=Q8, vocab=0, prefix_len=10)
    wl = synth.make_workload("moe_40rows", cfg, 40, 10, 104)
    _run(wl, 10)


def test_moe_int8_asym_experts_nine_rows(cuda):
    cfg = _moe(max_rows=9, fmt_attn=I8, fmt_dense=I8, fmt_shared=I8, fmt_routed=I8, vocab=0, n_shared=1,
               prefix_len=7)
    wl = synth.make_workload("moe_i8", cfg, 9, 10, 105)
    _run(wl, 10)


def test_moe_q4_shared_q4_routed_no_shared_dense_free(cuda):
    cfg = _moe(n_dense_layers=0, n_layers=2, n_shared=0, fmt_routed=Q4, vocab=0, prefix_len=3, max_rows=2,
               top_k=2, n_experts=8)
    wl = synth.make_workload("moe_noshared", cfg, 2, 12, 106)
    _run(wl, 12)


def test_moe_q4_both_with_lm_head_rows_12(cuda):
    cfg = _moe(fmt_shared=Q4, fmt_routed=Q4, max_rows=12, prefix_len=6)
    wl = synth.make_workload("moe_q4_lm", cfg, 12, 6, 107, prefix="prefill", n_prefill_embeds=3,
                             step_input="ids")
    _run(wl, 6)


def _wide(**kw):
    # hidden 2048: every projection needs several 16 KB stages per slab (Q8_0 QKV 2, Q4_0 expert
    # gate/up 2, shared down 3, LM head 4) and the 78-slot cache spans two attention stages
    base = dict(hidden=2048, n_heads=16, head_dim=128, n_layers=2, n_dense_layers=1, dense_inter=1024,
                n_experts=8, top_k=2, n_shared=2, expert_inter=1024, vocab=2000, fmt_attn=Q8, fmt_dense=Q8,
                fmt_shared=Q8, fmt_routed=Q4, prefix_len=70, ring_len=8, max_rows=3)
    base.update(kw)
    return synth.ModelConfig(**base)


def test_multi_chunk_slabs_q4_routed_q8_shared(cuda):
    wl = synth.make_workload("wide_q4r_q8s", _wide(), 3, 10, 108, step_input="ids")
    st = _run(wl, 10)
    assert st.id_checks >= 3 * 10


def test_multi_chunk_slabs_q8_routed_q4_shared(cuda):
    wl = synth.make_workload("wide_q8r_q4s", _wide(fmt_routed=Q8, fmt_shared=Q4, vocab=0), 3, 10, 109)
    _run(wl, 10)


def test_moe_uocr_prefill_three_chunks_then_greedy(cuda):
    """uocr_prefill against the oracle's prefill-by-decode: 100 embeddings (two
    chunks, 64 + 36 tokens) then 50 prompt ids (one ragged chunk) per row; every
    prefix key and value, the last prompt token's layer taps, logits and id, then
    greedy steps from that cache."""
    cfg = _moe(prefix_len=150, max_rows=3)
    wl = synth.make_workload("moe_prefill", cfg, 3, 6, 110, prefix="prefill", n_prefill_embeds=100,
                             step_input="ids")
    st = _run(wl, 6, lib_prefill=True)
    assert st.kv_checks >= 3 * cfg.n_layers + 3 * 6 * cfg.n_layers
    assert st.id_checks >= 3 * 7


def test_dense_uocr_prefill_with_sinks_int8_asym(cuda):
    """uocr_prefill of a dense decoder with attention sinks, int8-asymmetric
    weights and head_dim 64 (30 embeddings, then 10 prompt ids), then greedy
    steps through the ring."""
    cfg = _dense(fmt_attn=I8, fmt_dense=I8, use_sink=1, prefix_len=40, ring_len=16, max_rows=2, vocab=500)
    wl = synth.make_workload("dense_prefill_ring", cfg, 2, 5, 111, prefix="prefill", n_prefill_embeds=30,
                             step_input="ids")
    _run(wl, 5, lib_prefill=True)


# ---------------------------------------------------------------- INT8 KV cache
def _code_steps_small(st, frac=0.02):
    print(f"INT8 entries: {st.kv_codes} codes, {st.kv_code_steps} one step off")
    assert st.kv_codes > 0 and st.kv_code_steps <= frac * st.kv_codes


def test_int8_kv_dense_ring_wrap_sinks_head_dim_64(cuda):
    cfg = _dense(kv_int8=1, use_sink=1, fmt_attn=I8, fmt_dense=Q8)
    wl = synth.make_workload("i8kv_dense", cfg, 3, 20, 120)
    _code_steps_small(_run(wl, 20))


def test_int8_kv_moe_prefill_by_decode_then_greedy(cuda):
    wl = synth.make_workload("i8kv_moe_lm", _moe(kv_int8=1), 5, 10, 121, prefix="prefill", n_prefill_embeds=8,
                             step_input="ids")
    st = _run(wl, 10)
    assert st.id_checks >= 5 * 10
    _code_steps_small(st)


def test_int8_kv_moe_forty_rows_three_token_groups(cuda):
    cfg = _moe(kv_int8=1, max_rows=40, fmt_shared=Q4, vocab=0, prefix_len=10)
    wl = synth.make_workload("i8kv_moe_40rows", cfg, 40, 8, 122)
    _code_steps_small(_run(wl, 8))


def test_int8_kv_uocr_prefill_two_chunks(cuda):
    cfg = _moe(kv_int8=1, prefix_len=90, max_rows=2)
    wl = synth.make_workload("i8kv_prefill", cfg, 2, 5, 123, prefix="prefill", n_prefill_embeds=70,
                             step_input="ids")
    _code_steps_small(_run(wl, 5, lib_prefill=True))


# ---------------------------------------------------------------- group-64 blocks
G8, G4 = synth.Q8_0_G64, synth.Q4_0_G64


def test_group64_dense_q8_attention_q4_mlp_ring_wrap(cuda):
    cfg = _dense(fmt_attn=G8, fmt_dense=G4)
    wl = synth.make_workload("g64_dense", cfg, 3, 12, 130)
    st = _run(wl, 12)
    assert st.kv_checks == 12 * 2 * 3


def test_group64_moe_q4_routed_q8_shared_with_lm_head(cuda):
    cfg = _moe(fmt_attn=G8, fmt_dense=G8, fmt_shared=G8, fmt_routed=G4, max_rows=12)
    wl = synth.make_workload("g64_moe", cfg, 12, 8, 131, prefix="prefill", n_prefill_embeds=5, step_input="ids")
    st = _run(wl, 8)
    assert st.id_checks >= 12 * 8 and st.router_checks > 0


def test_group64_moe_both_q4_forty_rows(cuda):
    cfg = _moe(fmt_shared=G4, fmt_routed=G4, max_rows=40, vocab=0, prefix_len=9)
    wl = synth.make_workload("g64_moe40", cfg, 40, 6, 132)
    _run(wl, 6)


# ---------------------------------------------------------------- int8 activations
def test_int8_activations_dense_q8_attention_q4_mlp_ring_wrap(cuda):
    cfg = _dense(act_int8=1, fmt_attn=Q8, fmt_dense=Q4)
    wl = synth.make_workload("a8_dense", cfg, 3, 20, 140)
    st = _run(wl, 20)
    assert st.kv_checks == 20 * 2 * 3


def test_int8_activations_i8asym_sink_decoder_forty_rows(cuda):
    # three token groups (16, 16, 8) of the two-n-tile kernels; zero points corrected from code sums
    cfg = _dense(act_int8=1, fmt_attn=I8, fmt_dense=I8, use_sink=1, max_rows=40, prefix_len=9)
    wl = synth.make_workload("a8_sink40", cfg, 40, 8, 141)
    _run(wl, 8)


def test_int8_activations_six_rows_staged_once_q4_attention(cuda):
    # 4..8 rows: one 8-row token group quantised once per projection and copied by every CTA
    cfg = _dense(act_int8=1, fmt_attn=Q4, fmt_dense=I8, use_sink=1, max_rows=6, prefix_len=7)
    wl = synth.make_workload("a8_six", cfg, 6, 12, 145)
    _run(wl, 12)


def test_int8_activations_with_int8_kv_sink_decoder_single_row(cuda):
    cfg = _dense(act_int8=1, kv_int8=1, fmt_attn=I8, fmt_dense=I8, use_sink=1, max_rows=1, hidden=1024,
                 n_heads=8, head_dim=64, dense_inter=1024, n_layers=2, n_dense_layers=2, prefix_len=33)
    wl = synth.make_workload("a8_i8kv_sink", cfg, 1, 10, 142)
    _code_steps_small(_run(wl, 10))


def test_int8_activations_moe_prefill_by_decode_then_greedy(cuda):
    wl = synth.make_workload("a8_moe_lm", _moe(act_int8=1, max_rows=12), 12, 8, 143, prefix="prefill",
                             n_prefill_embeds=6, step_input="ids")
    st = _run(wl, 8)
    assert st.id_checks >= 12 * 8 and st.router_checks > 0


def test_int8_activations_group64_blocks(cuda):
    cfg = _dense(act_int8=1, fmt_attn=G8, fmt_dense=G4, max_rows=9)
    wl = synth.make_workload("a8_g64", cfg, 9, 10, 144)
    _run(wl, 10)


# ---------------------------------------------------------------- tensor-core experts
# The tcgen05 expert kernels (more than 16 rows, off by default) are switched on
# per context by UOCR_TC_EXPERTS=1, read when the context is created.
@pytest.fixture
def tc_experts(monkeypatch):
    monkeypatch.setenv("UOCR_TC_EXPERTS", "1")


def _layer_outputs(cfg, wl, tc, monkeypatch):
    import torch

    monkeypatch.setenv("UOCR_TC_EXPERTS", tc)
    ctx = make_ctx(wl)
    x = torch.from_numpy(np.ascontiguousarray(wl.step_x[0]).view(np.int16)).cuda()
    pos = torch.full((wl.rows,), cfg.prefix_len, dtype=torch.int32, device="cuda")
    y = torch.zeros((wl.rows, cfg.hidden), dtype=torch.float32, device="cuda")
    ctx.uocr_decode_step_embeds(wl.rows, x.data_ptr(), pos.data_ptr(), y.data_ptr())
    ctx.uocr_sync()
    out = y.cpu().numpy().astype(np.float64)
    ctx.close()
    return out


def test_tensor_core_experts_forty_rows_q4_routed_q8_shared(cuda, tc_experts):
    cfg = _moe(max_rows=40, vocab=0, prefix_len=10)
    wl = synth.make_workload("tcx_moe40", cfg, 40, 6, 150)
    st = _run(wl, 6)
    assert st.router_checks > 0 and st.grouping_checks > 0


def test_tensor_core_experts_q8_routed_q4_shared_two_token_groups_with_lm_head(cuda, tc_experts):
    cfg = _moe(fmt_routed=Q8, fmt_shared=Q4, max_rows=24)
    wl = synth.make_workload("tcx_moe24_lm", cfg, 24, 6, 151, prefix="prefill", n_prefill_embeds=5,
                             step_input="ids")
    st = _run(wl, 6)
    assert st.id_checks >= 24 * 6


def test_tensor_core_experts_run_and_agree_with_the_fragment_kernels(cuda, monkeypatch):
    cfg = _moe(max_rows=33, vocab=0, prefix_len=10)
    wl = synth.make_workload("tcx_ab", cfg, 33, 1, 152)
    on = _layer_outputs(cfg, wl, "1", monkeypatch)
    off = _layer_outputs(cfg, wl, "0", monkeypatch)
    # different kernels (the scale folded into the fp16 weight on the tensor cores):
    # not bit-identical, within the stated tolerance of each other
    assert np.any(on != off)
    rel = float(np.linalg.norm(on - off) / np.linalg.norm(off))
    assert rel <= 2e-3, rel


# ---------------------------------------------------------------- projector
@pytest.mark.parametrize("fmt,n", [(Q8, 40), (G4, 7), (I8, 33)])
def test_projector_against_the_oracle(cuda, fmt, n):
    torch = cuda
    import oracle

    cfg = _dense(proj_in=512, fmt_proj=fmt, max_rows=1)
    wl = synth.make_workload("proj", cfg, 1, 1, 133)
    ctx = make_ctx(wl)
    rng = np.random.default_rng(134)
    feats = rng.standard_normal((n, 512)).astype(np.float16)
    x = torch.from_numpy(feats.view(np.int16)).cuda()
    out = torch.zeros((n, cfg.hidden), dtype=torch.int16, device="cuda")
    ctx.uocr_project(n, x.data_ptr(), out.data_ptr())
    ctx.uocr_sync()
    got = out.cpu().numpy().view(np.float16).astype(np.float64)
    want = make_oracle(wl).project(feats.astype(np.float64))
    from parity import check_close
    e, m, _ = check_close("projector", got, want)
    print(f"\nprojector fmt {fmt} n {n}: rel-L2 {e:.2e} max-abs {m:.2e}")
    ctx.close()


# ---------------------------------------------------------------- tensor-core LM head
@pytest.mark.parametrize("rows", [20, 64])
def test_lm_head_on_tensor_cores_rows_above_16(cuda, rows):
    """Steps of more than 16 rows run the LM head as a tcgen05 GEMM (N = 32 or 64
    padded rows, vocabulary 1000: the last 128-row tile is ragged): logits and
    greedy ids against the oracle over several steps."""
    cfg = _dense(vocab=1000, max_rows=rows, n_layers=1, n_dense_layers=1)
    wl = synth.make_workload("tc_lm", cfg, rows, 4, 140, step_input="ids")
    st = _run(wl, 4)
    assert st.id_checks == rows * 4
