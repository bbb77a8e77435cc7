"""The scratch-free LM head entry point against the regular decode step.

uocr_lm_head_argmax_noalloc is for callers that may not allocate device
memory while they run (a serving loop whose memory belongs to a fixed pool, a
host framework that only lends the buffers it owns): it runs the same LM-head
+ argmax kernel as the decode step, with the kernel's scratch in a static
device array instead of the context arena.  Given the final hidden states of
a step it must reproduce that step's logits and ids bit for bit (the same
kernel over the same slabs in the same order), on two calls in a row (the
second call sees the scratch the first one left behind), with one token group
(12 rows) and with four (64 rows, the capacity of the scratch), with and
without a logits output.

This file is collected last on purpose; it passes alone in a fresh process and
after the other tests.
"""
import numpy as np
import pytest

from quantized_moe_decode_gb300 import binding, synth

from helpers import make_ctx

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("rows", [12, 64])
def test_noalloc_lm_head_matches_decode_step_twice(cuda, rows):
    torch = cuda
    cfg = synth.ModelConfig(hidden=256, n_heads=2, head_dim=128, n_layers=2, n_dense_layers=1, dense_inter=512,
                            n_experts=8, top_k=2, n_shared=1, expert_inter=128, vocab=1000,
                            fmt_attn=synth.Q8_0, fmt_dense=synth.Q8_0, fmt_shared=synth.Q8_0,
                            fmt_routed=synth.Q4_0, prefix_len=5, ring_len=8, max_rows=rows)
    wl = synth.make_workload("noalloc", cfg, rows, 2, 300, step_input="ids")
    ctx = make_ctx(wl)
    dev = torch.device("cuda")
    ids = torch.from_numpy(wl.first_ids).to(dev)
    pos = torch.full((rows,), wl.start_pos, dtype=torch.int32, device=dev)
    nxt = torch.zeros(rows, dtype=torch.int32, device=dev)
    lg = torch.zeros((rows, cfg.vocab), dtype=torch.float32, device=dev)
    nxt2 = torch.zeros(rows, dtype=torch.int32, device=dev)
    lg2 = torch.zeros((rows, cfg.vocab), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    device_before = torch.cuda.current_device()
    for call in range(2):
        ctx.uocr_decode_step(rows, ids.data_ptr(), pos.data_ptr(), nxt.data_ptr(), lg.data_ptr())
        ctx.uocr_sync()
        hidden = torch.from_numpy(ctx.uocr_debug_hidden(2 * cfg.n_layers - 1, rows)).to(dev)
        for with_logits in (True, False):
            lg2.fill_(float("nan"))
            nxt2.fill_(-1)
            ctx.uocr_lm_head_argmax_noalloc(rows, hidden.data_ptr(), nxt2.data_ptr(),
                                            lg2.data_ptr() if with_logits else 0, stream.cuda_stream)
            stream.synchronize()
            assert np.array_equal(nxt2.cpu().numpy(), nxt.cpu().numpy()), f"call {call} ids"
            if with_logits:
                assert np.array_equal(lg2.cpu().numpy(), lg.cpu().numpy()), f"call {call} logits"
            else:
                assert np.isnan(lg2.cpu().numpy()).all(), "logits written without a logits buffer"
        ids.copy_(nxt)
        pos += 1
    assert torch.cuda.current_device() == device_before
    with pytest.raises(binding.UocrError) as e:
        ctx.uocr_lm_head_argmax_noalloc(65, hidden.data_ptr(), nxt2.data_ptr(), 0, stream.cuda_stream)
    assert e.value.status == binding.UOCR_E_INVALID_ARG
    ctx.close()
