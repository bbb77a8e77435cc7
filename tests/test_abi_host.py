"""Host-side checks of the C ABI that need no GPU: the library builds, loads and
exports every function include/uocr.h declares, and config / budget errors are
reported before any device work."""
import os
import re

import pytest

from quantized_moe_decode_gb300 import binding, synth

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "uocr.h")


def _declared():
    txt = open(HEADER).read()
    return sorted(set(re.findall(r"^UOCR_API\s+[\w\s\*]+?\b(uocr_\w+)\(", txt, flags=re.M)))


def test_header_declares_the_binding_names():
    assert _declared() == sorted(binding.EXPORTED)


def test_library_exports_every_declared_symbol(libuocr):
    for name in _declared():
        assert hasattr(libuocr, name), name


def test_invalid_config_is_rejected_on_the_host(libuocr):
    cfg = synth.config_dense_layer()
    for bad in (dict(hidden=100), dict(head_dim=48), dict(max_rows=0), dict(max_rows=65), dict(ring_len=0),
                dict(n_dense_layers=5)):
        with pytest.raises(binding.UocrError) as e:
            binding.Context(cfg.replace(**bad))
        assert e.value.status == binding.UOCR_E_INVALID_ARG
    moe = synth.config_moe_layer()
    with pytest.raises(binding.UocrError) as e:
        binding.Context(moe.replace(top_k=9))
    assert e.value.status == binding.UOCR_E_INVALID_ARG
    with pytest.raises(binding.UocrError) as e:
        binding.Context(moe.replace(fmt_routed=synth.F16))
    assert e.value.status == binding.UOCR_E_INVALID_ARG
    # int8 activations multiply int8 weight codes: fp16 projections are refused
    for bad in (dict(act_int8=1, fmt_attn=synth.F16), dict(act_int8=1, fmt_dense=synth.F16), dict(act_int8=2)):
        with pytest.raises(binding.UocrError) as e:
            binding.Context(cfg.replace(**bad))
        assert e.value.status == binding.UOCR_E_INVALID_ARG


def test_budget_refusal_names_every_category(libuocr):
    with pytest.raises(binding.UocrError) as e:
        binding.Context(synth.config_full(), mem_budget=1 << 20)
    assert e.value.status == binding.UOCR_E_BUDGET
    for cat in ("weights", "kv_cache", "activations", "routing", "logits"):
        assert cat in str(e.value)
