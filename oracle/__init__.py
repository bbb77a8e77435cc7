"""Float64 CPU oracle of the quantized MoE decode step.

TEST INFRASTRUCTURE: only tests/, __graft_entry__.smoke() and bench.py's
cpu_baseline / reference leg may import, call or execute anything here.  It
shares no code with the CUDA library in quantized_moe_decode_gb300/ and never
imports it.
"""
from .model import (TIE_TOL, OracleModel, StepResult, act_quant, argmax_first, attend, attend_lse,  # noqa: F401
                    f16, group_by_expert, kv_dequant, kv_quant, project, rmsnorm, rope, route, ring_slot,
                    silu, swiglu, swiglu_rows)
from .quant import dequant, float32_is_exact  # noqa: F401
