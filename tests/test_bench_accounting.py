"""The algorithmic bytes behind bench.py's GB/s and roofline figures, pinned to
per-layer constants worked out by hand from the block formats (Q8_0: 32 codes
+ one fp16 scale = 34 bytes per 32 weights; Q4_0: 16 bytes of nibbles + one
fp16 scale = 18 bytes per 32 weights; fp16: 2 bytes per weight) and the
decoder's shapes (hidden 1280, 10 x 128 heads, dense MLP 3584, experts of
896, 64 routed experts, vocab 102400)."""
import bench
from quantized_moe_decode_gb300 import synth


def _weights_only(cfg, distinct):
    # no rows and no positions: only the weight terms remain
    return bench.class_bytes(cfg, 0, [], distinct)


def test_attention_dense_router_and_lm_head_weights():
    cfg = synth.config_full(max_rows=8)
    b = _weights_only(cfg, {l: 0 for l in range(1, 12)})
    assert b["qkv"][0] + b["o_proj"][0] == 6_963_200  # (3 + 1) * 1280 * 1280 * 34 / 32
    assert b["mlp_gate_up"][0] + b["mlp_down"][0] == 14_622_720  # 3 * 3584 * 1280 * 34 / 32
    assert b["router"][0] == 163_840  # 64 * 1280 * 2
    assert b["lm_head_argmax"][0] == 262_144_000  # 102400 * 1280 * 2
    assert len(b["qkv"]) == 12 and len(b["router"]) == 11 and len(b["mlp_gate_up"]) == 1


def test_expert_weights_scale_with_the_experts_picked():
    cfg = synth.config_stress(max_rows=64)  # every expert Q4_0, shared ones too
    one = _weights_only(cfg, {l: 1 for l in range(1, 12)})
    none = _weights_only(cfg, {l: 0 for l in range(1, 12)})
    per_expert = (one["expert_gate_up"][0] + one["expert_down"][0]
                  - none["expert_gate_up"][0] - none["expert_down"][0])
    assert per_expert == 1_935_360  # 3 * 896 * 1280 * 18 / 32
    assert none["expert_gate_up"][0] + none["expert_down"][0] == 3_870_720  # two shared, Q4_0
    full = synth.config_full(max_rows=8)  # shared experts Q8_0
    z = _weights_only(full, {l: 0 for l in range(1, 12)})
    assert z["expert_gate_up"][0] + z["expert_down"][0] == 7_311_360  # 2 * 3 * 896 * 1280 * 34 / 32


def test_kv_bytes_per_row_and_layer_follow_the_valid_slots():
    cfg = synth.config_full(max_rows=8)  # P = 288, ring 128, K and V of 10 x 128 fp16
    d = {l: 0 for l in range(1, 12)}

    def att(p):
        return bench.class_bytes(cfg, 1, [p], d)["attention"][0]

    # inside the prefix: p + 1 slots; in the ring: P + min(p - P + 1, 128) slots; 5120 bytes per slot
    assert att(11) - att(10) == 5120
    assert att(300) - att(288) == 12 * 5120
    assert att(288 + 127) - att(288 + 126) == 5120
    assert att(288 + 500) == att(288 + 127)  # the ring is full: the count stops growing
