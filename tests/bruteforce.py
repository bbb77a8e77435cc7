"""A second, independent statement of the decode step in scalar Python.

Used only to pin the oracle on tiny shapes.  Activations are rounded to fp16
where the method stores them (normalised matmul inputs, cached keys and
values, attention output, SwiGLU activations).  It parses the weight blocks with
``struct`` byte by byte, keeps the KV history as a dict keyed by absolute
position (no slots, no ring arithmetic), applies the ring rule as a mask on
absolute positions, and spells every sum as a loop.  It shares nothing with
oracle/ beyond the meaning of the canonical bytes.
"""
from __future__ import annotations

import math
import struct


def _half(b0, b1):
    return struct.unpack("<e", bytes([b0, b1]))[0]


def decode_rows(t):
    """Canonical blob -> list of rows (lists of Python floats)."""
    b = bytes(t.blob.tobytes())
    rows, cols, fmt = t.rows, t.cols, t.fmt
    out = []
    if fmt == 0:
        vals = struct.unpack("<%de" % (rows * cols), b)
        return [list(vals[r * cols:(r + 1) * cols]) for r in range(rows)]
    size = {1: 34, 2: 18, 3: 36, 4: 66, 5: 34}[fmt]
    group = {1: 32, 2: 32, 3: 32, 4: 64, 5: 64}[fmt]
    pos = 0
    for _ in range(rows):
        row = []
        for _ in range(cols // group):
            blk = b[pos:pos + size]
            pos += size
            if fmt in (1, 4):
                d = _half(blk[0], blk[1])
                for j in range(group):
                    q = blk[2 + j]
                    q = q - 256 if q >= 128 else q
                    row.append(d * q)
            elif fmt in (2, 5):
                d = _half(blk[0], blk[1])
                half = group // 2
                codes = [blk[2 + j] % 16 for j in range(half)] + [blk[2 + j] // 16 for j in range(half)]
                for q in codes:
                    row.append(d * (q - 8))
            else:
                s = _half(blk[0], blk[1])
                z = _half(blk[2], blk[3])
                for j in range(32):
                    row.append(s * (blk[4 + j] - z))
        out.append(row)
    return out


def h16(v):
    """Round a Python float to fp16 (nearest even) through struct's half format."""
    return struct.unpack("<e", struct.pack("<e", v))[0]


def matvec(W, x):
    return [sum(W[n][k] * x[k] for k in range(len(x))) for n in range(len(W))]


def norm(x, w, eps):
    ms = sum(v * v for v in x) / len(x)
    r = 1.0 / math.sqrt(ms + eps)
    return [x[i] * r * w[i] for i in range(len(x))]


def rot(v, p, theta):
    """Rotate-half RoPE as complex multiplication of (v[i] + i*v[i+D/2])."""
    D = len(v)
    h = D // 2
    out = [0.0] * D
    for i in range(h):
        z = complex(v[i], v[i + h]) * complex(math.cos(p * theta ** (-2.0 * i / D)),
                                              math.sin(p * theta ** (-2.0 * i / D)))
        out[i], out[i + h] = z.real, z.imag
    return out


def mlp(x, g, u, d):
    a = [0.0] * len(g)
    gx, ux = matvec(g, x), matvec(u, x)
    for i in range(len(g)):
        a[i] = h16(gx[i] / (1.0 + math.exp(-gx[i])) * ux[i])  # activations stored in fp16
    return matvec(d, a)


class BruteModel:
    def __init__(self, cfg, tensors, rows, kv_prefix=None, sinks=None):
        self.cfg = cfg
        self.W = {(t.kind, t.layer, t.expert): decode_rows(t) for t in tensors}
        self.rows = rows
        self.sinks = sinks
        # hist[row][layer] = {position: (k_heads, v_heads)}
        self.hist = [[{} for _ in range(cfg.n_layers)] for _ in range(rows)]
        if kv_prefix is not None:
            for l, (k, v) in enumerate(kv_prefix):
                for r in range(rows):
                    for p in range(cfg.prefix_len):
                        self.hist[r][l][p] = ([[float(a) for a in k[r, h, p]] for h in range(cfg.n_heads)],
                                              [[float(a) for a in v[r, h, p]] for h in range(cfg.n_heads)])

    def vec(self, kind, layer=0, expert=0):
        return self.W[(kind, layer, expert)][0]

    def mat(self, kind, layer=0, expert=0):
        return self.W[(kind, layer, expert)]

    def step_row(self, r, p, x):
        cfg = self.cfg
        nh, D, P, R = cfg.n_heads, cfg.head_dim, cfg.prefix_len, cfg.ring_len
        layers_out = []
        for l in range(cfg.n_layers):
            xn = [h16(a) for a in norm(x, self.vec(3, l), cfg.rms_eps)]
            q = matvec(self.mat(4, l), xn)
            k = matvec(self.mat(5, l), xn)
            v = matvec(self.mat(6, l), xn)
            qh = [rot(q[h * D:(h + 1) * D], p, cfg.rope_theta) for h in range(nh)]
            kh = [[h16(a) for a in rot(k[h * D:(h + 1) * D], p, cfg.rope_theta)] for h in range(nh)]
            vh = [[h16(a) for a in v[h * D:(h + 1) * D]] for h in range(nh)]
            self.hist[r][l][p] = (kh, vh)
            keep = [pp for pp in sorted(self.hist[r][l]) if pp <= p and (pp < P or pp > p - R)]
            att = []
            for h in range(nh):
                logits = [sum(qh[h][i] * self.hist[r][l][pp][0][h][i] for i in range(D)) / math.sqrt(D)
                          for pp in keep]
                vals = [self.hist[r][l][pp][1][h] for pp in keep]
                if cfg.use_sink:
                    logits.append(float(self.sinks[l][h]))
                    vals.append([0.0] * D)
                m = max(logits)
                e = [math.exp(a - m) for a in logits]
                z = sum(e)
                att += [h16(sum(e[j] * vals[j][i] for j in range(len(e))) / z) for i in range(D)]
            o = matvec(self.mat(7, l), att)
            hh = [x[i] + o[i] for i in range(len(x))]
            hn = [h16(a) for a in norm(hh, self.vec(8, l), cfg.rms_eps)]
            if l < cfg.n_dense_layers or cfg.n_experts == 0:
                m = mlp(hn, self.mat(9, l), self.mat(10, l), self.mat(11, l))
                y = [hh[i] + m[i] for i in range(len(hh))]
            else:
                lg = matvec(self.mat(12, l), hn)
                # top-k by repeated selection of the first maximum among the rest
                chosen = []
                for _ in range(cfg.top_k):
                    best = None
                    for e in range(cfg.n_experts):
                        if e in chosen:
                            continue
                        if best is None or lg[e] > lg[best]:
                            best = e
                    chosen.append(best)
                mx = max(lg)
                pe = [math.exp(a - mx) for a in lg]
                tot = sum(pe)
                prob = [a / tot for a in pe]
                sel = sum(prob[e] for e in chosen)
                y = list(hh)
                for e in chosen:
                    m = mlp(hn, self.mat(16, l, e), self.mat(17, l, e), self.mat(18, l, e))
                    for i in range(len(y)):
                        y[i] += prob[e] / sel * m[i]
                for s in range(cfg.n_shared):
                    m = mlp(hn, self.mat(13, l, s), self.mat(14, l, s), self.mat(15, l, s))
                    for i in range(len(y)):
                        y[i] += m[i]
            layers_out.append(y)
            x = y
        logits = None
        if cfg.vocab:
            xn = [h16(a) for a in norm(x, self.vec(1), cfg.rms_eps)]
            logits = matvec(self.mat(2), xn)
        return layers_out, logits

    def step(self, positions, ids=None, x=None):
        outs = []
        for r in range(self.rows):
            if x is None:
                xr = list(self.mat(0)[int(ids[r])])
            else:
                xr = [float(a) for a in x[r]]
            outs.append(self.step_row(r, int(positions[r]), xr))
        return outs
