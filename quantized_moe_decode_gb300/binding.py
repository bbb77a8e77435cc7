"""ctypes binding of libuocr.so: the C ABI of include/uocr.h under the same names.

Argument marshalling only: every step of the decode path runs in the CUDA
library.  Loading fails loudly when the library is missing; there is no
fallback.  Device buffers are passed as integer addresses (for example
``torch.Tensor.data_ptr()``).
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
# UOCR_LIB selects another build of the same library (tuning variants)
LIB_PATH = os.environ.get("UOCR_LIB") or os.path.join(_PKG, "libuocr.so")

UOCR_OK, UOCR_E_INVALID_ARG, UOCR_E_OOM, UOCR_E_BUDGET, UOCR_E_FORMAT = 0, 1, 2, 3, 4
UOCR_E_STATE, UOCR_E_CUDA, UOCR_E_POSITION, UOCR_E_TOKEN, UOCR_E_TIMEOUT = 5, 6, 7, 8, 9
STATUS_NAMES = {0: "OK", 1: "E_INVALID_ARG", 2: "E_OOM", 3: "E_BUDGET", 4: "E_FORMAT", 5: "E_STATE",
                6: "E_CUDA", 7: "E_POSITION", 8: "E_TOKEN", 9: "E_TIMEOUT"}

EXPORTED = ["uocr_create", "uocr_destroy", "uocr_load_weights", "uocr_kv_write_prefix", "uocr_kv_write",
            "uocr_kv_read",
            "uocr_set_sinks", "uocr_decode_step", "uocr_decode_step_embeds", "uocr_decode_step_host",
            "uocr_prefill", "uocr_generate", "uocr_kv_reset", "uocr_sync", "uocr_last_error", "uocr_memory_report",
            "uocr_debug_hidden", "uocr_debug_router", "uocr_debug_router_logits", "uocr_profile",
            "uocr_lm_head_argmax_noalloc", "uocr_debug_wait_probe", "uocr_kv_read_i8", "uocr_kv_write_i8", "uocr_project"]


class uocr_config(C.Structure):
    _fields_ = [(n, C.c_int32) for n in (
        "hidden", "n_heads", "head_dim", "n_layers", "n_dense_layers", "dense_inter", "n_experts", "top_k",
        "n_shared", "expert_inter", "vocab", "fmt_attn", "fmt_dense", "fmt_shared", "fmt_routed",
        "prefix_len", "ring_len", "max_rows", "use_sink")] + [
        ("rms_eps", C.c_float), ("rope_theta", C.c_float), ("mem_budget", C.c_uint64),
        ("stream", C.c_void_p), ("device", C.c_int32), ("use_graphs", C.c_int32), ("kv_int8", C.c_int32),
        ("proj_in", C.c_int32), ("fmt_proj", C.c_int32), ("act_int8", C.c_int32)]


class uocr_tensor(C.Structure):
    _fields_ = [("kind", C.c_int32), ("layer", C.c_int32), ("expert", C.c_int32), ("format", C.c_int32),
                ("rows", C.c_int32), ("cols", C.c_int32), ("data", C.c_void_p), ("bytes", C.c_uint64)]


class uocr_mem_report(C.Structure):
    _fields_ = [(n, C.c_uint64) for n in ("weights", "kv_cache", "activations", "routing", "logits", "total")]


_lib = None


def load(path: str = LIB_PATH):
    """Load libuocr.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} not found: build it with quantized_moe_decode_gb300.build.build()")
    lib = C.CDLL(path)
    P, I, U64 = C.c_void_p, C.c_int32, C.c_uint64
    sig = {
        "uocr_create": ([C.POINTER(uocr_config), C.POINTER(P)], I),
        "uocr_destroy": ([P], None),
        "uocr_load_weights": ([P, C.POINTER(uocr_tensor), C.c_size_t], I),
        "uocr_kv_write_prefix": ([P, I, I, P, P, I, I], I),
        "uocr_kv_read": ([P, I, I, I, I, P, P], I),
        "uocr_kv_write": ([P, I, I, I, I, P, P], I),
        "uocr_set_sinks": ([P, P], I),
        "uocr_decode_step": ([P, I, P, P, P, P], I),
        "uocr_decode_step_embeds": ([P, I, P, P, P, P, P, P], I),
        "uocr_prefill": ([P, I, P, P, I, I, P, P], I),
        "uocr_decode_step_host": ([P, I, P, P, P], I),
        "uocr_generate": ([P, I, P, P, I, P], I),
        "uocr_kv_reset": ([P, I, I], I),
        "uocr_sync": ([P], I),
        "uocr_last_error": ([P], C.c_char_p),
        "uocr_memory_report": ([P, C.POINTER(uocr_mem_report)], I),
        "uocr_debug_hidden": ([P, I, I, P], I),
        "uocr_debug_router": ([P, I, I, P, P, P, P, P], I),
        "uocr_debug_router_logits": ([P, I, I, P], I),
        "uocr_profile": ([P, I, I, P, P, P, C.POINTER(C.c_char_p), C.POINTER(C.c_float), C.POINTER(I)], I),
        "uocr_lm_head_argmax_noalloc": ([P, I, P, P, P, P], I),
        "uocr_debug_wait_probe": ([P, I], I),
        "uocr_kv_read_i8": ([P, I, I, I, I, P, P, P, P], I),
        "uocr_kv_write_i8": ([P, I, I, I, I, P, P, P, P], I),
        "uocr_project": ([P, I, P, P], I),
    }
    for name, (args, res) in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    _lib = lib
    return lib


class UocrError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


def make_config(cfg, *, max_rows=None, mem_budget=0, stream=0, device=0, use_graphs=1) -> uocr_config:
    """uocr_config from any object with the model-config attribute names."""
    c = uocr_config()
    for n in ("hidden", "n_heads", "head_dim", "n_layers", "n_dense_layers", "dense_inter", "n_experts",
              "top_k", "n_shared", "expert_inter", "vocab", "fmt_attn", "fmt_dense", "fmt_shared",
              "fmt_routed", "prefix_len", "ring_len", "max_rows", "use_sink"):
        setattr(c, n, int(getattr(cfg, n)))
    if max_rows is not None:
        c.max_rows = int(max_rows)
    c.rms_eps = float(cfg.rms_eps)
    c.rope_theta = float(cfg.rope_theta)
    c.mem_budget = int(mem_budget)
    c.stream = int(stream) or None
    c.device = int(device)
    c.use_graphs = int(use_graphs)
    c.kv_int8 = int(getattr(cfg, "kv_int8", 0))
    c.proj_in = int(getattr(cfg, "proj_in", 0))
    c.fmt_proj = int(getattr(cfg, "fmt_proj", 1))
    c.act_int8 = int(getattr(cfg, "act_int8", 0))
    return c


class Context:
    """Owns one uocr_ctx; methods map one-to-one onto the C calls."""

    def __init__(self, cfg, **kw):
        self.lib = load()
        self.cfg = cfg
        self._c = make_config(cfg, **kw)
        h = C.c_void_p()
        st = self.lib.uocr_create(C.byref(self._c), C.byref(h))
        if st != UOCR_OK:
            raise UocrError(st, self.lib.uocr_last_error(None).decode())
        self.h = h

    def _ck(self, st):
        if st != UOCR_OK:
            raise UocrError(st, self.lib.uocr_last_error(self.h).decode())

    def close(self):
        if getattr(self, "h", None):
            self.lib.uocr_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- loading
    def uocr_load_weights(self, tensors):
        arr = (uocr_tensor * len(tensors))()
        keep = []
        for i, t in enumerate(tensors):
            b = np.ascontiguousarray(t.blob)
            keep.append(b)
            arr[i] = uocr_tensor(t.kind, t.layer, t.expert, t.fmt, t.rows, t.cols, b.ctypes.data, b.nbytes)
        self._ck(self.lib.uocr_load_weights(self.h, arr, len(tensors)))

    def uocr_kv_write_prefix(self, row, layer, k, v, start=0):
        k = np.ascontiguousarray(k, dtype=np.float16)
        v = np.ascontiguousarray(v, dtype=np.float16)
        self._ck(self.lib.uocr_kv_write_prefix(self.h, row, layer, k.ctypes.data, v.ctypes.data, start,
                                               k.shape[1]))

    def uocr_kv_write(self, row, layer, slot0, k, v):
        """k, v: fp16 [n_heads][n][head_dim] written to slots [slot0, slot0+n)."""
        k = np.ascontiguousarray(k, dtype=np.float16)
        v = np.ascontiguousarray(v, dtype=np.float16)
        self._ck(self.lib.uocr_kv_write(self.h, row, layer, slot0, k.shape[1], k.ctypes.data, v.ctypes.data))

    def uocr_kv_read(self, row, layer, slot0, n):
        nh, D = self.cfg.n_heads, self.cfg.head_dim
        k = np.empty((nh, n, D), np.float16)
        v = np.empty((nh, n, D), np.float16)
        self._ck(self.lib.uocr_kv_read(self.h, row, layer, slot0, n, k.ctypes.data, v.ctypes.data))
        return k, v

    def uocr_kv_read_i8(self, row, layer, slot0, n):
        """INT8 cache entries: (k codes int8 [nh][n][D], k scales fp32 [nh][n], v codes, v scales)."""
        nh, D = self.cfg.n_heads, self.cfg.head_dim
        kc = np.empty((nh, n, D), np.int8)
        vc = np.empty((nh, n, D), np.int8)
        ks = np.empty((nh, n), np.float32)
        vs = np.empty((nh, n), np.float32)
        self._ck(self.lib.uocr_kv_read_i8(self.h, row, layer, slot0, n, kc.ctypes.data, ks.ctypes.data,
                                          vc.ctypes.data, vs.ctypes.data))
        return kc, ks, vc, vs

    def uocr_kv_write_i8(self, row, layer, slot0, kc, ks, vc, vs):
        """Write INT8 cache entries as given: codes [nh][n][D], scales [nh][n]."""
        kc = np.ascontiguousarray(kc, np.int8)
        vc = np.ascontiguousarray(vc, np.int8)
        ks = np.ascontiguousarray(ks, np.float32)
        vs = np.ascontiguousarray(vs, np.float32)
        self._ck(self.lib.uocr_kv_write_i8(self.h, row, layer, slot0, kc.shape[1], kc.ctypes.data, ks.ctypes.data,
                                           vc.ctypes.data, vs.ctypes.data))

    def uocr_set_sinks(self, sinks):
        s = np.ascontiguousarray(sinks, dtype=np.float32)
        self._ck(self.lib.uocr_set_sinks(self.h, s.ctypes.data))

    # -- steps (device addresses)
    def uocr_decode_step(self, rows, ids_ptr, pos_ptr, next_ptr, logits_ptr=0):
        self._ck(self.lib.uocr_decode_step(self.h, rows, ids_ptr, pos_ptr, next_ptr, logits_ptr or None))

    def uocr_decode_step_embeds(self, rows, x_ptr, pos_ptr, y_ptr=0, next_ptr=0, logits_ptr=0, y_f16_ptr=0):
        self._ck(self.lib.uocr_decode_step_embeds(self.h, rows, x_ptr, pos_ptr, y_ptr or None, y_f16_ptr or None,
                                                  next_ptr or None, logits_ptr or None))

    def uocr_prefill(self, row, n, start_pos, ids_ptr=0, x_ptr=0, next_ptr=0, logits_ptr=0):
        """Prefill n positions of cache row `row` from device token ids or fp16 hidden vectors."""
        self._ck(self.lib.uocr_prefill(self.h, row, ids_ptr or None, x_ptr or None, n, start_pos, next_ptr or None,
                                       logits_ptr or None))

    def uocr_project(self, n, feats_ptr, out_ptr):
        """Projector: device fp16 features [n][proj_in] -> device fp16 [n][hidden]."""
        self._ck(self.lib.uocr_project(self.h, n, feats_ptr, out_ptr))

    def uocr_debug_wait_probe(self, issue_copy):
        self._ck(self.lib.uocr_debug_wait_probe(self.h, int(issue_copy)))

    def uocr_decode_step_host(self, rows, ids, pos):
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        pos = np.ascontiguousarray(pos, dtype=np.int32)
        out = np.empty(rows, np.int32)
        self._ck(self.lib.uocr_decode_step_host(self.h, rows, ids.ctypes.data, pos.ctypes.data, out.ctypes.data))
        return out

    def uocr_generate(self, rows, ids_ptr, pos_ptr, n_steps, out_ptr):
        self._ck(self.lib.uocr_generate(self.h, rows, ids_ptr, pos_ptr, n_steps, out_ptr))

    def uocr_lm_head_argmax_noalloc(self, rows, hidden_ptr, next_ptr, logits_ptr=0, stream=0):
        self._ck(self.lib.uocr_lm_head_argmax_noalloc(self.h, rows, hidden_ptr, next_ptr, logits_ptr or None,
                                                      stream or None))

    def uocr_kv_reset(self, row=-1, keep_prefix=1):
        self._ck(self.lib.uocr_kv_reset(self.h, row, keep_prefix))

    def uocr_sync(self):
        self._ck(self.lib.uocr_sync(self.h))

    def uocr_memory_report(self) -> dict:
        r = uocr_mem_report()
        self._ck(self.lib.uocr_memory_report(self.h, C.byref(r)))
        return {n: int(getattr(r, n)) for n, _ in r._fields_}

    def uocr_debug_hidden(self, tap, rows):
        out = np.empty((rows, self.cfg.hidden), np.float32)
        self._ck(self.lib.uocr_debug_hidden(self.h, tap, rows, out.ctypes.data))
        return out

    def uocr_debug_router(self, layer, rows):
        k, E = self.cfg.top_k, self.cfg.n_experts
        idx = np.empty((rows, k), np.int32)
        w = np.empty((rows, k), np.float32)
        count = np.empty(E, np.int32)
        offset = np.empty(E + 1, np.int32)
        perm = np.empty(rows * k, np.int32)
        self._ck(self.lib.uocr_debug_router(self.h, layer, rows, idx.ctypes.data, w.ctypes.data,
                                            count.ctypes.data, offset.ctypes.data, perm.ctypes.data))
        return dict(idx=idx, w=w, count=count, offset=offset, perm=perm)

    def uocr_debug_router_logits(self, layer, rows):
        out = np.empty((rows, self.cfg.n_experts), np.float32)
        self._ck(self.lib.uocr_debug_router_logits(self.h, layer, rows, out.ctypes.data))
        return out

    def uocr_profile(self, rows, input_kind, ids_ptr, x_ptr, pos_ptr, cap=32):
        names = (C.c_char_p * cap)()
        ms = (C.c_float * cap)()
        n = C.c_int32(cap)
        self._ck(self.lib.uocr_profile(self.h, rows, input_kind, ids_ptr or None, x_ptr or None, pos_ptr, names,
                                       ms, C.byref(n)))
        return {names[i].decode(): float(ms[i]) for i in range(min(n.value, cap))}


def load_workload(ctx: Context, wl, chunk: int = 64):
    """Upload a synthetic workload's weights, cached prefix and sinks."""
    ts = wl.tensors
    for i in range(0, len(ts), chunk):
        ctx.uocr_load_weights(ts[i:i + chunk])
    if wl.kv_prefix is not None:
        for l in range(wl.cfg.n_layers):
            for r in range(wl.rows):
                k, v = wl.kv_prefix.get(l, r)
                ctx.uocr_kv_write_prefix(r, l, k, v, 0)
    if wl.sinks is not None:
        ctx.uocr_set_sinks(wl.sinks)
