"""C ABI behaviour on the GPU: chained generation, the host-buffer entry point,
graphs against eager launches, determinism, device-side status reporting and
host-side refusals.  All through the C ABI."""
import numpy as np
import pytest

from quantized_moe_decode_gb300 import binding, synth

from helpers import make_ctx

pytestmark = pytest.mark.gpu


def _cfg(**kw):
    base = dict(hidden=256, n_heads=2, head_dim=128, n_layers=3, n_dense_layers=1, dense_inter=512,
                n_experts=16, top_k=4, n_shared=2, expert_inter=128, vocab=1000, fmt_attn=synth.Q8_0,
                fmt_dense=synth.Q8_0, fmt_shared=synth.Q8_0, fmt_routed=synth.Q4_0, prefix_len=6, ring_len=8,
                max_rows=4)
    base.update(kw)
    return synth.ModelConfig(**base)


def _wl(seed=200, **kw):
    return synth.make_workload("api", _cfg(**kw), 4, 8, seed, step_input="ids")


def _greedy_steps(ctx, torch, wl, n):
    ids = torch.from_numpy(wl.first_ids).cuda()
    pos = torch.full((wl.rows,), wl.start_pos, dtype=torch.int32, device="cuda")
    nxt = torch.zeros(wl.rows, dtype=torch.int32, device="cuda")
    out = []
    for s in range(n):
        ctx.uocr_decode_step(wl.rows, ids.data_ptr(), pos.data_ptr(), nxt.data_ptr())
        ctx.uocr_sync()
        out.append(nxt.cpu().numpy().copy())
        ids.copy_(nxt)
        pos += 1
    return np.stack(out)


def test_generate_equals_step_loop_and_host_entry_point(cuda):
    torch = cuda
    wl = _wl()
    a = make_ctx(wl)
    ref = _greedy_steps(a, torch, wl, 12)
    b = make_ctx(wl)
    ids = torch.from_numpy(wl.first_ids).cuda()
    pos = torch.full((wl.rows,), wl.start_pos, dtype=torch.int32, device="cuda")
    out = torch.zeros((12, wl.rows), dtype=torch.int32, device="cuda")
    b.uocr_generate(wl.rows, ids.data_ptr(), pos.data_ptr(), 12, out.data_ptr())
    b.uocr_sync()
    assert np.array_equal(out.cpu().numpy(), ref)
    c = make_ctx(wl)
    got = []
    cur = wl.first_ids.copy()
    for s in range(12):
        cur = c.uocr_decode_step_host(wl.rows, cur, np.full(wl.rows, wl.start_pos + s, np.int32))
        got.append(cur)
    assert np.array_equal(np.stack(got), ref)
    for x in (a, b, c):
        x.close()


def test_graph_and_eager_launches_are_bit_identical_and_deterministic(cuda):
    torch = cuda
    wl = _wl(seed=201)
    runs = []
    for graphs in (1, 0, 1):
        ctx = make_ctx(wl, use_graphs=graphs)
        ids = torch.from_numpy(wl.first_ids).cuda()
        pos = torch.full((wl.rows,), wl.start_pos, dtype=torch.int32, device="cuda")
        nxt = torch.zeros(wl.rows, dtype=torch.int32, device="cuda")
        lg = torch.zeros((wl.rows, wl.cfg.vocab), dtype=torch.float32, device="cuda")
        outs = []
        for s in range(4):
            ctx.uocr_decode_step(wl.rows, ids.data_ptr(), pos.data_ptr(), nxt.data_ptr(), lg.data_ptr())
            ctx.uocr_sync()
            outs.append(lg.cpu().numpy().copy())
            ids.copy_(nxt)
            pos += 1
        runs.append(np.stack(outs))
        ctx.close()
    assert np.array_equal(runs[0], runs[1])
    assert np.array_equal(runs[0], runs[2])


def test_device_status_reports_bad_token_and_position(cuda):
    torch = cuda
    wl = _wl(seed=202)
    ctx = make_ctx(wl)
    ids = torch.tensor([1, 2, wl.cfg.vocab, 3], dtype=torch.int32, device="cuda")
    pos = torch.full((4,), wl.start_pos, dtype=torch.int32, device="cuda")
    nxt = torch.zeros(4, dtype=torch.int32, device="cuda")
    ctx.uocr_decode_step(4, ids.data_ptr(), pos.data_ptr(), nxt.data_ptr())
    with pytest.raises(binding.UocrError) as e:
        ctx.uocr_sync()
    assert e.value.status == binding.UOCR_E_TOKEN
    ctx.uocr_sync()  # cleared
    ids[2] = 5
    pos[1] = -3
    ctx.uocr_decode_step(4, ids.data_ptr(), pos.data_ptr(), nxt.data_ptr())
    with pytest.raises(binding.UocrError) as e:
        ctx.uocr_sync()
    assert e.value.status == binding.UOCR_E_POSITION
    ctx.close()


def test_host_side_refusals(cuda):
    torch = cuda
    wl = _wl(seed=203)
    ctx = binding.Context(wl.cfg, max_rows=wl.rows)
    ids = torch.zeros(4, dtype=torch.int32, device="cuda")
    with pytest.raises(binding.UocrError) as e:  # no weights yet
        ctx.uocr_decode_step(4, ids.data_ptr(), ids.data_ptr(), ids.data_ptr())
    assert e.value.status == binding.UOCR_E_STATE
    t = wl.tensors[1]
    bad = synth.Tensor(t.kind, t.layer, t.expert, t.fmt, t.rows, t.cols, t.blob[:-1])
    with pytest.raises(binding.UocrError) as e:
        ctx.uocr_load_weights([bad])
    assert e.value.status == binding.UOCR_E_FORMAT
    wrong_fmt = synth.Tensor(t.kind, t.layer, t.expert, synth.Q4_0, t.rows, t.cols, t.blob)
    with pytest.raises(binding.UocrError) as e:
        ctx.uocr_load_weights([wrong_fmt])
    assert e.value.status == binding.UOCR_E_FORMAT
    binding.load_workload(ctx, wl)
    for bad_rows in (5, 0, -1):  # above max_rows, an empty step, a negative count
        with pytest.raises(binding.UocrError) as e:
            ctx.uocr_decode_step(bad_rows, ids.data_ptr(), ids.data_ptr(), ids.data_ptr())
        assert e.value.status == binding.UOCR_E_INVALID_ARG
    rep = ctx.uocr_memory_report()
    assert rep["total"] >= rep["weights"] + rep["kv_cache"] > 0
    ctx.close()


def test_kv_reset_keeps_prefix_and_clears_ring(cuda):
    torch = cuda
    wl = _wl(seed=204)
    ctx = make_ctx(wl)
    _greedy_steps(ctx, torch, wl, 3)
    P = wl.cfg.prefix_len
    k_before, _ = ctx.uocr_kv_read(1, 0, 0, P + 3)
    assert np.any(k_before[:, P:] != 0)
    ctx.uocr_kv_reset(1, keep_prefix=1)
    k_after, v_after = ctx.uocr_kv_read(1, 0, 0, P + 3)
    assert np.array_equal(k_after[:, :P], k_before[:, :P])
    assert not np.any(k_after[:, P:]) and not np.any(v_after[:, P:])
    ctx.close()


def test_bounded_wait_reports_timeout_and_context_stays_usable(cuda):
    """The TMA waits poll an mbarrier with an iteration limit.  The probe runs
    that wait with a short limit: with its 16-byte copy issued the wait
    succeeds; with the copy never issued it runs out, uocr_sync reports
    UOCR_E_TIMEOUT once, and the context still decodes."""
    torch = cuda
    wl = _wl(seed=205)
    ctx = make_ctx(wl)
    ctx.uocr_debug_wait_probe(1)
    ctx.uocr_sync()  # the copy landed: no status
    ctx.uocr_debug_wait_probe(0)
    with pytest.raises(binding.UocrError) as e:
        ctx.uocr_sync()
    assert e.value.status == binding.UOCR_E_TIMEOUT
    ctx.uocr_sync()  # cleared
    ref = make_ctx(wl)
    assert np.array_equal(_greedy_steps(ctx, torch, wl, 3), _greedy_steps(ref, torch, wl, 3))
    ctx.close()
    ref.close()


def test_embeds_step_fp16_output_is_the_rounded_fp32_output(cuda):
    torch = cuda
    cfg = _cfg(vocab=0)
    wl = synth.make_workload("api_x", cfg, 4, 2, 206)
    ctx = make_ctx(wl)
    x = torch.from_numpy(np.ascontiguousarray(wl.step_x[0]).view(np.int16)).cuda()
    pos = torch.full((4,), wl.start_pos, dtype=torch.int32, device="cuda")
    y = torch.zeros((4, cfg.hidden), dtype=torch.float32, device="cuda")
    y16 = torch.zeros((4, cfg.hidden), dtype=torch.int16, device="cuda")
    ctx.uocr_decode_step_embeds(4, x.data_ptr(), pos.data_ptr(), y_ptr=y.data_ptr(), y_f16_ptr=y16.data_ptr())
    ctx.uocr_sync()
    got = y16.cpu().numpy().view(np.float16)
    assert np.array_equal(got, y.cpu().numpy().astype(np.float16))
    ctx.close()


def test_prefill_refusals(cuda):
    torch = cuda
    wl = _wl(seed=207)
    ctx = make_ctx(wl)
    ids = torch.zeros(8, dtype=torch.int32, device="cuda")
    x = torch.zeros((8, wl.cfg.hidden), dtype=torch.int16, device="cuda")
    SL = wl.cfg.prefix_len + wl.cfg.ring_len
    for kw, st in ((dict(ids_ptr=ids.data_ptr(), x_ptr=x.data_ptr()), binding.UOCR_E_INVALID_ARG),
                   (dict(), binding.UOCR_E_INVALID_ARG)):
        with pytest.raises(binding.UocrError) as e:
            ctx.uocr_prefill(0, 4, 0, **kw)
        assert e.value.status == st
    for row, n, start in ((-1, 4, 0), (4, 4, 0), (0, 0, 0), (0, 4, -1), (0, 4, SL - 3)):
        with pytest.raises(binding.UocrError) as e:
            ctx.uocr_prefill(row, n, start, ids_ptr=ids.data_ptr())
        assert e.value.status == binding.UOCR_E_INVALID_ARG, (row, n, start)
    ctx.uocr_prefill(0, 3, SL - 3, ids_ptr=ids.data_ptr())  # the last ring slots, no wrap
    ctx.uocr_sync()
    ctx.close()


def test_int8_cache_prefix_quantised_exactly_and_entry_io(cuda):
    """A written prefix is fp16 on both sides, so the INT8 entries (codes and
    scales, decided in fp32) equal the oracle's bit for bit; exact entries
    written with uocr_kv_write_i8 read back unchanged; uocr_kv_read gives
    scale * code in fp16; the fp16 cache refuses the INT8 calls."""
    import oracle

    cfg = _cfg(kv_int8=1, prefix_len=40, head_dim=64, n_heads=4)
    wl = _wl(seed=208, kv_int8=1, prefix_len=40, head_dim=64, n_heads=4)
    ctx = make_ctx(wl)
    nh, D = cfg.n_heads, cfg.head_dim
    for r in range(wl.rows):
        for l in range(cfg.n_layers):
            k, v = wl.kv_prefix.get(l, r)
            kc, ks, vc, vs = ctx.uocr_kv_read_i8(r, l, 0, cfg.prefix_len)
            okc, oks = oracle.kv_quant(k)
            ovc, ovs = oracle.kv_quant(v)
            assert np.array_equal(kc, okc) and np.array_equal(ks, oks), (r, l)
            assert np.array_equal(vc, ovc) and np.array_equal(vs, ovs), (r, l)
    kd, vd = ctx.uocr_kv_read(1, 1, 3, 5)
    kc, ks, vc, vs = ctx.uocr_kv_read_i8(1, 1, 3, 5)
    assert np.array_equal(kd, (ks[..., None] * kc.astype(np.float32)).astype(np.float16))
    rng = np.random.default_rng(3)
    ck = rng.integers(-127, 128, size=(nh, 4, D)).astype(np.int8)
    sk = rng.uniform(0.01, 0.1, size=(nh, 4)).astype(np.float32)
    ctx.uocr_kv_write_i8(2, 0, cfg.prefix_len + 1, ck, sk, -ck, 2 * sk)
    got = ctx.uocr_kv_read_i8(2, 0, cfg.prefix_len + 1, 4)
    assert np.array_equal(got[0], ck) and np.array_equal(got[1], sk)
    assert np.array_equal(got[2], -ck) and np.array_equal(got[3], 2 * sk)
    ctx.close()
    f16 = make_ctx(_wl(seed=209))
    with pytest.raises(binding.UocrError) as e:
        f16.uocr_kv_read_i8(0, 0, 0, 1)
    assert e.value.status == binding.UOCR_E_STATE
    f16.close()
