"""Seeded synthetic inputs for the quantized MoE decode step.

This module only draws random numbers and encodes them into the canonical
weight block formats; it holds none of the decode arithmetic (no dequantisation,
no matmul, no attention).  Both the CUDA library (through the C ABI) and the
float64 oracle consume exactly the bytes produced here.

Recipe (one ``numpy.random.default_rng(seed)`` PCG64 stream per workload, drawn
in this fixed order: weights, then cached prefix / prefix inputs, then sinks,
then per-step inputs):

* linear weights ~ N(0, 0.02) (float32 draw), then block-encoded:
  Q8_0   blocks of 32: d = amax/127 (fp16), q = round(x/d) in [-127, 127]
  Q4_0   blocks of 32: d = m/-8 with m the signed value of largest magnitude,
         q = clamp(round(x/d) + 8, 0, 15) packed low nibbles first
  I8ASYM blocks of 32: s = (max-min)/255 (fp16), z = round(-min/s) (fp16),
         q = clamp(round(x/s) + z, 0, 255)
  The block definitions follow the decode-step statement: Q8_0 -> d*q,
  Q4_0 -> d*(q-8), int8-asymmetric -> s*(q-z), one fp16 scale per 32 values.
* RMSNorm weights 1 + N(0, 0.05) fp16; embedding and LM head N(0, 0.02) fp16;
  router N(0, router_std) fp16.
* cached prefix keys/values ~ N(0, 1) fp16 (treated as already rotated);
  attention sinks ~ N(0, 1) fp32 per layer and head;
  step inputs x ~ N(0, 1) fp16; token ids uniform in [0, vocab).
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass, field

import numpy as np

# Weight formats (values match uocr_format in include/uocr.h).
F16, Q8_0, Q4_0, I8ASYM = 0, 1, 2, 3
# group-64 variants of Q8_0 / Q4_0 (the Metal page's group size)
Q8_0_G64, Q4_0_G64 = 4, 5
FMT_NAMES = {F16: "f16", Q8_0: "q8_0", Q4_0: "q4_0", I8ASYM: "i8asym", Q8_0_G64: "q8_0_g64",
             Q4_0_G64: "q4_0_g64"}
BLOCK = 32
GROUP = {Q8_0: 32, Q4_0: 32, I8ASYM: 32, Q8_0_G64: 64, Q4_0_G64: 64}
BLOCK_BYTES = {Q8_0: 34, Q4_0: 18, I8ASYM: 36, Q8_0_G64: 66, Q4_0_G64: 34}

# Tensor kinds (values match uocr_tensor_kind in include/uocr.h).
T_EMBED, T_FINAL_NORM, T_LM_HEAD = 0, 1, 2
T_ATTN_NORM, T_WQ, T_WK, T_WV, T_WO, T_MLP_NORM = 3, 4, 5, 6, 7, 8
T_GATE, T_UP, T_DOWN = 9, 10, 11
T_ROUTER = 12
T_SHARED_GATE, T_SHARED_UP, T_SHARED_DOWN = 13, 14, 15
T_EXPERT_GATE, T_EXPERT_UP, T_EXPERT_DOWN = 16, 17, 18
T_PROJ, T_PROJ_BIAS = 19, 20


@dataclass
class ModelConfig:
    hidden: int
    n_heads: int
    head_dim: int
    n_layers: int
    n_dense_layers: int
    dense_inter: int
    n_experts: int = 0
    top_k: int = 0
    n_shared: int = 0
    expert_inter: int = 0
    vocab: int = 0
    fmt_attn: int = Q8_0
    fmt_dense: int = Q8_0
    fmt_shared: int = Q8_0
    fmt_routed: int = Q4_0
    prefix_len: int = 0
    ring_len: int = 128
    max_rows: int = 1
    use_sink: int = 0
    rms_eps: float = 1e-6
    rope_theta: float = 10000.0
    router_std: float = 0.02
    kv_int8: int = 0  # INT8 KV cache (one scale per head vector) instead of fp16
    act_int8: int = 0  # dynamic int8 activations (groups of 32) on the dense projections
    proj_in: int = 0  # projector input width (visual features; 0 = no projector)
    fmt_proj: int = Q8_0

    @property
    def moe(self) -> bool:
        return self.n_experts > 0 and self.n_layers > self.n_dense_layers

    def is_dense(self, layer: int) -> bool:
        return layer < self.n_dense_layers or self.n_experts == 0

    def replace(self, **kw) -> "ModelConfig":
        return dataclasses.replace(self, **kw)


@dataclass
class Tensor:
    kind: int
    layer: int
    expert: int
    fmt: int
    rows: int
    cols: int
    blob: np.ndarray  # uint8, canonical bytes

    @property
    def nbytes(self) -> int:
        return int(self.blob.nbytes)


@dataclass
class Workload:
    """A model, its weights and the inputs of every decode step."""

    name: str
    cfg: ModelConfig
    rows: int
    steps: int
    seed: int
    tensors: list = field(default_factory=list)
    # cached prefix: kv_prefix[layer] = (k, v) with k, v fp16 [rows, heads, P, D]
    # (a KVPrefix: drawn lazily, per (layer, row))
    kv_prefix: "KVPrefix | None" = None
    sinks: np.ndarray | None = None  # fp32 [layers, heads]
    # prefix built by running decode steps (prefill-by-decode):
    prefill_embeds: np.ndarray | None = None  # fp16 [rows, n_embed, H]
    prefill_ids: np.ndarray | None = None  # int32 [rows, n_ids]
    # per-step inputs: either hidden vectors or (first) token ids
    step_x: np.ndarray | None = None  # fp16 [steps, rows, H]
    first_ids: np.ndarray | None = None  # int32 [rows]
    start_pos: int = 0  # position of the first decode step

    def positions(self, step: int) -> np.ndarray:
        return np.full(self.rows, self.start_pos + step, dtype=np.int32)


# ---------------------------------------------------------------- encoders
def _fp16_bytes(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a.astype(np.float16)).view(np.uint8)


def encode_q8_0(x: np.ndarray, group: int = BLOCK) -> np.ndarray:
    n, k = x.shape
    xb = x.reshape(n, k // group, group).astype(np.float32)
    amax = np.abs(xb).max(axis=-1)
    d = (amax / 127.0).astype(np.float16)
    df = d.astype(np.float32)
    inv = np.divide(1.0, df, out=np.zeros_like(df), where=df != 0)
    q = np.clip(np.rint(xb * inv[..., None]), -127, 127).astype(np.int8)
    out = np.empty((n, k // group, 2 + group), np.uint8)
    out[..., 0:2] = d.view(np.uint8).reshape(n, k // group, 2)
    out[..., 2:] = q.view(np.uint8)
    return out.reshape(-1)


def encode_q4_0(x: np.ndarray, group: int = BLOCK) -> np.ndarray:
    n, k = x.shape
    xb = x.reshape(n, k // group, group).astype(np.float32)
    am = np.abs(xb).argmax(axis=-1)
    m = np.take_along_axis(xb, am[..., None], axis=-1)[..., 0]
    d = (m / -8.0).astype(np.float16)
    df = d.astype(np.float32)
    inv = np.divide(1.0, df, out=np.zeros_like(df), where=df != 0)
    q = np.clip(np.rint(xb * inv[..., None]) + 8, 0, 15).astype(np.uint8)
    half = group // 2
    out = np.empty((n, k // group, 2 + half), np.uint8)
    out[..., 0:2] = d.view(np.uint8).reshape(n, k // group, 2)
    # element j < half -> low nibble of byte j; element j >= half -> high nibble of byte j-half
    out[..., 2:] = q[..., :half] | (q[..., half:] << 4)
    return out.reshape(-1)


def encode_i8asym(x: np.ndarray) -> np.ndarray:
    n, k = x.shape
    xb = x.reshape(n, k // BLOCK, BLOCK).astype(np.float32)
    mn = xb.min(axis=-1)
    mx = xb.max(axis=-1)
    s = ((mx - mn) / 255.0).astype(np.float16)
    sf = s.astype(np.float32)
    inv = np.divide(1.0, sf, out=np.zeros_like(sf), where=sf != 0)
    z = np.clip(np.rint(-mn * inv), 0, 255).astype(np.float16)
    q = np.clip(np.rint(xb * inv[..., None]) + z.astype(np.float32)[..., None], 0, 255).astype(np.uint8)
    out = np.empty((n, k // BLOCK, 36), np.uint8)
    out[..., 0:2] = s.view(np.uint8).reshape(n, k // BLOCK, 2)
    out[..., 2:4] = z.view(np.uint8).reshape(n, k // BLOCK, 2)
    out[..., 4:] = q
    return out.reshape(-1)


def encode(x: np.ndarray, fmt: int) -> np.ndarray:
    if fmt == F16:
        return _fp16_bytes(x).reshape(-1)
    if fmt == Q8_0:
        return encode_q8_0(x)
    if fmt == Q4_0:
        return encode_q4_0(x)
    if fmt == I8ASYM:
        return encode_i8asym(x)
    if fmt == Q8_0_G64:
        return encode_q8_0(x, 64)
    if fmt == Q4_0_G64:
        return encode_q4_0(x, 64)
    raise ValueError(f"unknown format {fmt}")


def blob_bytes(fmt: int, rows: int, cols: int) -> int:
    if fmt == F16:
        return rows * cols * 2
    return rows * (cols // GROUP[fmt]) * BLOCK_BYTES[fmt]


# ---------------------------------------------------------------- weights
def _linear(rng, kind, layer, expert, fmt, rows, cols, std=0.02) -> Tensor:
    x = rng.standard_normal((rows, cols), dtype=np.float32) * np.float32(std)
    return Tensor(kind, layer, expert, fmt, rows, cols, encode(x, fmt))


def _norm(rng, kind, layer, h) -> Tensor:
    w = 1.0 + 0.05 * rng.standard_normal(h, dtype=np.float32)
    return Tensor(kind, layer, 0, F16, 1, h, _fp16_bytes(w).reshape(-1))


def make_weights(cfg: ModelConfig, rng: np.random.Generator) -> list:
    H, S = cfg.hidden, cfg.n_heads * cfg.head_dim
    ts = []
    if cfg.vocab:
        ts.append(_linear(rng, T_EMBED, 0, 0, F16, cfg.vocab, H))
    for l in range(cfg.n_layers):
        ts.append(_norm(rng, T_ATTN_NORM, l, H))
        for kind in (T_WQ, T_WK, T_WV):
            ts.append(_linear(rng, kind, l, 0, cfg.fmt_attn, S, H))
        ts.append(_linear(rng, T_WO, l, 0, cfg.fmt_attn, H, S))
        ts.append(_norm(rng, T_MLP_NORM, l, H))
        if cfg.is_dense(l):
            I = cfg.dense_inter
            ts.append(_linear(rng, T_GATE, l, 0, cfg.fmt_dense, I, H))
            ts.append(_linear(rng, T_UP, l, 0, cfg.fmt_dense, I, H))
            ts.append(_linear(rng, T_DOWN, l, 0, cfg.fmt_dense, H, I))
        else:
            I = cfg.expert_inter
            ts.append(_linear(rng, T_ROUTER, l, 0, F16, cfg.n_experts, H, std=cfg.router_std))
            for s in range(cfg.n_shared):
                ts.append(_linear(rng, T_SHARED_GATE, l, s, cfg.fmt_shared, I, H))
                ts.append(_linear(rng, T_SHARED_UP, l, s, cfg.fmt_shared, I, H))
                ts.append(_linear(rng, T_SHARED_DOWN, l, s, cfg.fmt_shared, H, I))
            for e in range(cfg.n_experts):
                ts.append(_linear(rng, T_EXPERT_GATE, l, e, cfg.fmt_routed, I, H))
                ts.append(_linear(rng, T_EXPERT_UP, l, e, cfg.fmt_routed, I, H))
                ts.append(_linear(rng, T_EXPERT_DOWN, l, e, cfg.fmt_routed, H, I))
    if cfg.vocab:
        ts.append(_norm(rng, T_FINAL_NORM, 0, H))
        ts.append(_linear(rng, T_LM_HEAD, 0, 0, F16, cfg.vocab, H))
    if cfg.proj_in:  # drawn last: configs without a projector keep their streams
        ts.append(_linear(rng, T_PROJ, 0, 0, cfg.fmt_proj, H, cfg.proj_in))
        ts.append(_linear(rng, T_PROJ_BIAS, 0, 0, F16, 1, H))
    return ts


def _f16_normal(rng, shape) -> np.ndarray:
    return rng.standard_normal(shape, dtype=np.float32).astype(np.float16)


class KVPrefix:
    """Cached prefix keys/values ~ N(0,1) fp16, drawn lazily per (layer, row).

    A pool of 2**24 N(0,1) fp16 samples is drawn once from the workload seed;
    the keys (values) of one (layer, row) are the window of nh*P*D consecutive
    pool samples (cyclically) starting at an offset drawn from a generator
    seeded by (seed, layer, row, 0 or 1).  A (layer, row) therefore never
    depends on how many rows the workload has, one row can be drawn without the
    others, and the gigabytes of cache that long prefixes at many rows need
    cost a copy instead of a fresh draw.
    """

    POOL = 1 << 24

    def __init__(self, seed: int, n_layers: int, rows: int, nh: int, P: int, D: int):
        self.seed, self.n_layers, self.rows = seed, n_layers, rows
        self.shape = (nh, P, D)
        self._pool = None

    def _window(self, layer: int, row: int, which: int) -> np.ndarray:
        if self._pool is None:
            rng = np.random.default_rng([self.seed, 0x4B56])
            self._pool = _f16_normal(rng, (self.POOL,))
        n = int(np.prod(self.shape))
        start = int(np.random.default_rng([self.seed, layer, row, which]).integers(0, self.POOL))
        idx_end = start + n
        if idx_end <= self.POOL:
            flat = self._pool[start:idx_end].copy()
        else:  # wrap around the pool (as often as needed)
            reps = (idx_end + self.POOL - 1) // self.POOL
            flat = np.concatenate([self._pool[start:]] + [self._pool] * (reps - 2) +
                                  [self._pool[:idx_end - (reps - 1) * self.POOL]])
        return flat.reshape(self.shape)

    def get(self, layer: int, row: int):
        """(k, v) fp16 [nh, P, D] of one row of one layer."""
        return self._window(layer, row, 0), self._window(layer, row, 1)

    def subset(self, rows) -> list:
        """Per layer (k, v) fp16 [len(rows), nh, P, D] for the given rows."""
        out = []
        for l in range(self.n_layers):
            kv = [self.get(l, r) for r in rows]
            out.append((np.stack([a for a, _ in kv]), np.stack([b for _, b in kv])))
        return out

    def __len__(self) -> int:
        return self.n_layers

    def __getitem__(self, layer: int):
        kv = [self.get(layer, r) for r in range(self.rows)]
        return np.stack([a for a, _ in kv]), np.stack([b for _, b in kv])

    def __iter__(self):
        return (self[l] for l in range(self.n_layers))


def make_workload(name: str, cfg: ModelConfig, rows: int, steps: int, seed: int, *,
                  prefix: str = "cached", n_prefill_embeds: int = 0,
                  step_input: str = "x") -> Workload:
    """Draw a workload.

    prefix: "cached"  -> cfg.prefix_len cached K/V per row and layer ~ N(0,1);
            "prefill" -> prefix built by decode steps over n_prefill_embeds
                         fp16 embeddings then (prefix_len - n_prefill_embeds)
                         token ids; decoding then starts at prefix_len.
    step_input: "x" -> fresh hidden vector per step; "ids" -> first token ids
                (greedy continuation afterwards).
    """
    assert rows <= cfg.max_rows
    rng = np.random.default_rng(seed)
    wl = Workload(name=name, cfg=cfg, rows=rows, steps=steps, seed=seed)
    wl.tensors = make_weights(cfg, rng)
    P, nh, D, H = cfg.prefix_len, cfg.n_heads, cfg.head_dim, cfg.hidden
    if prefix == "cached":
        wl.kv_prefix = KVPrefix(seed, cfg.n_layers, rows, nh, P, D)
    elif prefix == "prefill":
        assert 0 <= n_prefill_embeds <= P
        wl.prefill_embeds = _f16_normal(rng, (rows, n_prefill_embeds, H))
        wl.prefill_ids = rng.integers(0, cfg.vocab, size=(rows, P - n_prefill_embeds)).astype(np.int32)
    else:
        raise ValueError(prefix)
    if cfg.use_sink:
        wl.sinks = rng.standard_normal((cfg.n_layers, nh)).astype(np.float32)
    if step_input == "x":
        wl.step_x = _f16_normal(rng, (steps, rows, H))
    elif step_input == "ids":
        if prefix != "prefill":
            wl.first_ids = rng.integers(0, cfg.vocab, size=rows).astype(np.int32)
    else:
        raise ValueError(step_input)
    wl.start_pos = P
    return wl


# ---------------------------------------------------------------- the five workloads
DEEPSEEK_OCR = dict(hidden=1280, n_heads=10, head_dim=128, n_dense_layers=1,
                    dense_inter=3584, n_experts=64, top_k=6, n_shared=2,
                    expert_inter=896, vocab=102400, ring_len=128)


def config_dense_layer() -> ModelConfig:
    """One dense decoder layer, batch 1, 64 cached tokens, Q8_0 everywhere."""
    return ModelConfig(hidden=1280, n_heads=10, head_dim=128, n_layers=1, n_dense_layers=1,
                       dense_inter=3584, fmt_attn=Q8_0, fmt_dense=Q8_0, prefix_len=64,
                       ring_len=128, max_rows=1)


def config_moe_layer() -> ModelConfig:
    """One MoE decoder layer, batch 1, 289 cached tokens + 128-slot ring."""
    return ModelConfig(hidden=1280, n_heads=10, head_dim=128, n_layers=1, n_dense_layers=0,
                       dense_inter=0, n_experts=64, top_k=6, n_shared=2, expert_inter=896,
                       vocab=0, fmt_attn=Q8_0, fmt_shared=Q4_0, fmt_routed=Q4_0,
                       prefix_len=289, ring_len=128, max_rows=1)


def config_full(max_rows: int = 8) -> ModelConfig:
    """12-layer decoder, Q8_0 attention/dense/shared, Q4_0 routed, fp16 LM head."""
    return ModelConfig(n_layers=12, fmt_attn=Q8_0, fmt_dense=Q8_0, fmt_shared=Q8_0,
                       fmt_routed=Q4_0, prefix_len=288, max_rows=max_rows, **DEEPSEEK_OCR)


def config_sink(T: int, max_rows: int = 64) -> ModelConfig:
    """18-layer dense decoder with attention sinks, int8-asymmetric weights."""
    return ModelConfig(hidden=1024, n_heads=8, head_dim=64, n_layers=18, n_dense_layers=18,
                       dense_inter=4096, fmt_attn=I8ASYM, fmt_dense=I8ASYM, prefix_len=T,
                       ring_len=128, max_rows=max_rows, use_sink=1)


def config_stress(max_rows: int = 64) -> ModelConfig:
    """The 12-layer decoder at 64 rows, 2048 cached tokens, all experts Q4_0."""
    return ModelConfig(n_layers=12, fmt_attn=Q8_0, fmt_dense=Q8_0, fmt_shared=Q4_0,
                       fmt_routed=Q4_0, prefix_len=2048, max_rows=max_rows,
                       router_std=float(1.0 / np.sqrt(1280.0)), **DEEPSEEK_OCR)


def workload(name: str, steps: int | None = None, rows: int | None = None, T: int = 350) -> Workload:
    """The named workloads; `steps`/`rows` override the default counts."""
    if name == "dense_layer_b1":
        return make_workload(name, config_dense_layer(), rows or 1, steps or 1, 0)
    if name == "moe_layer_b1":
        return make_workload(name, config_moe_layer(), rows or 1, steps or 300, 1)
    if name == "full_b8":
        r = rows or 8
        return make_workload(name, config_full(max_rows=r), r, steps or 200, 2,
                             prefix="prefill", n_prefill_embeds=256, step_input="ids")
    if name == "full_b8_g64":  # the full decoder with the Metal page's group-64 blocks
        r = rows or 8
        cfg = config_full(max_rows=r).replace(fmt_attn=Q8_0_G64, fmt_dense=Q8_0_G64, fmt_shared=Q8_0_G64,
                                              fmt_routed=Q4_0_G64)
        return make_workload(name, cfg, r, steps or 200, 2, prefix="prefill", n_prefill_embeds=256,
                             step_input="ids")
    if name == "sink":
        r = rows or 1
        return make_workload(f"sink_r{r}_T{T}", config_sink(T, max_rows=r), r, steps or 32, 3)
    if name == "stress_b64":
        r = rows or 64
        return make_workload(name, config_stress(max_rows=r), r, steps or 128, 4,
                             step_input="ids")
    raise KeyError(name)
