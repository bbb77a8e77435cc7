"""Glue between the seeded workloads, the library context and the oracle."""
from __future__ import annotations

import numpy as np

import oracle
from quantized_moe_decode_gb300 import binding


def make_ctx(wl, **kw):
    ctx = binding.Context(wl.cfg, max_rows=wl.rows, **kw)
    binding.load_workload(ctx, wl)
    return ctx


def make_oracle(wl, rows=None, cache="float64"):
    rows = list(range(wl.rows)) if rows is None else list(rows)
    kv = None if wl.kv_prefix is None else wl.kv_prefix.subset(rows)
    return oracle.OracleModel(wl.cfg, wl.tensors, len(rows), kv_prefix=kv, sinks=wl.sinks, cache=cache,
                              kv_int8=bool(wl.cfg.kv_int8), act_int8=bool(getattr(wl.cfg, "act_int8", 0)))
