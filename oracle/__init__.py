"""CPU oracle of the S2-Pro Dual-AR frame decode — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s cpu_baseline leg may
import this package.  It shares no code with the CUDA path (``dual_ar_tts_gb300``) and
never imports it.

The arithmetic lives in ``s2_oracle.c`` (plain fp32 C); this module loads it with ctypes
and writes out, in Python, the generation loop that strings the pieces together:

* sem_mask and min_tokens_before_end — s2.cpp analysis ch.06 "Fast-AR codebook decoding and
  the generation main loop" §5 and §5.3;
* the frame loop (sample -> repetition-aware resample -> clamp -> 9 Fast-AR calls -> store
  -> step -> sample) — ch.06 §5.1, §5.2 and ch.02 "Overall architecture and Dual-AR data
  flow" §3.3-§3.5;
* repetition-aware sampling (RAS) — ch.06 §6; draw order — Mizuoto "Fish Speech" engine page,
  "parity with upstream";
* result compaction codes[cb * n_frames + f] — ch.06 §8.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libs2oracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile ``s2_oracle.c`` with plain gcc (-O2, OpenMP over independent outputs)."""
    src = os.path.join(_HERE, "s2_oracle.c")
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(src):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                               "-std=gnu11", src, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class Dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("dim", "n_layer", "n_head", "n_kv_head", "head_dim", "ffn", "vocab",
                                            "sem_begin", "sem_end", "im_end", "n_codebooks", "codebook_size")] + \
               [(n, ctypes.c_float) for n in ("sem_scale", "norm_eps", "rope_base")] + \
               [(n, ctypes.c_int) for n in ("qk_norm", "rope_table_bf16", "fast_dim", "fast_n_layer", "fast_n_head",
                                            "fast_n_kv_head", "fast_head_dim", "fast_ffn", "fast_window",
                                            "has_fast_project_in", "weight_dtype", "kv_dtype")]


def dims_struct(d: dict) -> Dims:
    s = Dims()
    for name, _ in Dims._fields_:
        setattr(s, name, d[name])
    return s


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            vp, i32, f32, f64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_double
            sig = {
                "or_rmsnorm": (None, [vp, i32, vp, f32, vp]),
                "or_rope": (None, [vp, i32, i32, f64, i32]),
                "or_gqa_head_map": (None, [i32, i32, vp]),
                "or_attention": (None, [vp, vp, vp, i32, i32, i32, i32, i32, vp]),
                "or_weight_count": (i32, [ctypes.POINTER(Dims)]),
                "or_new": (vp, [ctypes.POINTER(Dims), vp, i32, i32]),
                "or_free": (None, [vp]),
                "or_pos": (i32, [vp]),
                "or_set_pos": (i32, [vp, i32]),
                "or_embed": (None, [vp, vp, vp]),
                "or_prefill": (i32, [vp, vp, i32, vp, vp]),
                "or_step": (i32, [vp, vp, vp, vp]),
                "or_extend": (i32, [vp, vp, i32, vp, vp]),
                "or_fast_forward": (i32, [vp, vp, vp, i32, vp, vp]),
                "or_kv_io": (i32, [vp, i32, i32, i32, vp, vp, i32]),
                "or_draw": (i32, [vp, vp, i32, f32, f32, i32, vp, vp]),
                "or_kv_set_f16": (i32, [vp, i32, i32, vp, vp]),
                "or_head": (i32, [vp, vp, vp, vp]),
                "or_e4m3_value": (f64, [i32]),
                "or_e4m3_encode": (i32, [f32]),
                "or_quant_e4m3": (None, [vp, ctypes.c_longlong, i32, vp, vp]),
                "or_bind_e4m3": (i32, [vp, i32, vp, vp, i32]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


# ------------------------------------------------------------------ primitives

def rmsnorm(x, w=None, eps=1e-6):
    x = _f32(x)
    out = np.empty_like(x)
    wv = None if w is None else _f32(w)
    _load().or_rmsnorm(x.ctypes.data, x.size, None if wv is None else wv.ctypes.data, eps, out.ctypes.data)
    return out


def rope(x, pos, base=1e6, table_bf16=True):
    v = _f32(x).copy()
    _load().or_rope(v.ctypes.data, v.size, int(pos), float(base), int(bool(table_bf16)))
    return v


def gqa_head_map(hq, hkv):
    m = np.empty(hq, np.int32)
    _load().or_gqa_head_map(hq, hkv, m.ctypes.data)
    return m


def attention(q, K, V, n=None):
    """q [Hq][hd]; K, V [Hkv][S][hd]; attends slots 0..n-1 (default all)."""
    q, K, V = _f32(q), _f32(K), _f32(V)
    hq, hd = q.shape
    hkv, S, _ = K.shape
    out = np.empty_like(q)
    _load().or_attention(q.ctypes.data, K.ctypes.data, V.ctypes.data, hq, hkv, hd, S, S if n is None else n,
                         out.ctypes.data)
    return out


def draw(logits, temperature, top_p, top_k, E, ids=None):
    """Returns (token, diag[7]); see ``or_draw`` in s2_oracle.c."""
    lg = _f32(logits)
    e = _f32(E)
    assert e.size >= top_k
    diag = np.zeros(7, np.float32)
    idv = None if ids is None else _i32(ids)
    tok = _load().or_draw(lg.ctypes.data, None if idv is None else idv.ctypes.data, lg.size, float(temperature),
                          float(top_p), int(top_k), e.ctypes.data, diag.ctypes.data)
    return int(tok), diag


# ---------------------------------------------------------------- the session

# ------------------------------------------------------------------ e4m3 weights

def e4m3_value(code: int) -> float:
    """Value of an e4m3 code (OCP 8-bit float E4M3: bias 7, 3 mantissa bits, subnormals m*2^-9)."""
    return _load().or_e4m3_value(int(code))


def e4m3_encode(x: float) -> int:
    """Nearest e4m3 code of a finite fp32 x (ties to even mantissa; magnitudes >= 448 -> 448)."""
    return _load().or_e4m3_encode(float(x))


def quant_e4m3(w_bf16):
    """bf16 bit patterns [rows][cols] -> (uint8 codes [rows][cols], fp32 scales [rows]):
    scale = max|row| / 448 in fp32, code = e4m3(w / scale) (fp32 division); zero rows -> 0, 0."""
    w = np.ascontiguousarray(w_bf16, dtype=np.uint16)
    rows, cols = (w.shape[0], int(np.prod(w.shape[1:]))) if w.ndim > 1 else (1, w.shape[0])
    codes = np.empty((rows, cols), np.uint8)
    scales = np.empty(rows, np.float32)
    _load().or_quant_e4m3(w.ctypes.data, rows, cols, codes.ctypes.data, scales.ctypes.data)
    return codes, scales


def projection_indices(d: dict):
    """Table indices of the projection matrices (wqkv, wo, w1, w3, w2 of every layer of both
    transformers, fast_project_in when present, fast_output)."""
    out = []
    for l in range(d["n_layer"]):
        out += [3 + 9 * l + f for f in (1, 4, 6, 7, 8)]
    base = 3 + 9 * d["n_layer"]
    if d["has_fast_project_in"]:
        out.append(base)
    out.append(base + 3)
    for l in range(d["fast_n_layer"]):
        out += [base + 4 + 9 * l + f for f in (1, 4, 6, 7, 8)]
    return out


def quantize_projections(d: dict, weights):
    """{table index: (codes, scales)} for every projection of a bf16 weight table."""
    return {i: quant_e4m3(weights[i]) for i in projection_indices(d)}


class Session:
    """One stream of the oracle: weights (host arrays, table order) + its own fp32 KV cache.

    With ``quant`` ({table index: (codes, scales)}, see ``quantize_projections``) those entries
    are read as scale[row] * e4m3_value(code) instead of the bf16 matrix."""

    def __init__(self, d: dict, weights, slots: int, quant=None):
        lib = _load()
        self.d = d
        self._dims = dims_struct(d)
        n = lib.or_weight_count(ctypes.byref(self._dims))
        if n != len(weights):
            raise ValueError(f"weight table has {len(weights)} entries, oracle expects {n}")
        self._keep = [None if w is None else np.ascontiguousarray(w) for w in weights]
        self._ptrs = (ctypes.c_void_p * n)(*[None if w is None else w.ctypes.data for w in self._keep])
        self._h = lib.or_new(ctypes.byref(self._dims), self._ptrs, n, int(slots))
        if not self._h:
            raise MemoryError("oracle session allocation failed")
        self.slots = slots
        self._quant = quant
        for i, (codes, scales) in (quant or {}).items():
            if lib.or_bind_e4m3(self._h, int(i), codes.ctypes.data, scales.ctypes.data, int(codes.shape[-1])):
                raise ValueError(f"binding e4m3 weights to table entry {i} failed")

    def close(self):
        if getattr(self, "_h", None):
            _load().or_free(self._h)
            self._h = None

    __del__ = close

    @property
    def pos(self):
        return _load().or_pos(self._h)

    def set_pos(self, p):
        if _load().or_set_pos(self._h, int(p)):
            raise ValueError("position out of range")

    def embed(self, vals):
        v = _i32(vals)
        x = np.empty(self.d["dim"], np.float32)
        _load().or_embed(self._h, v.ctypes.data, x.ctypes.data)
        return x

    def prefill(self, tokens):
        t = _i32(tokens)
        logits = np.empty(self.d["vocab"], np.float32)
        hidden = np.empty(self.d["dim"], np.float32)
        rc = _load().or_prefill(self._h, t.ctypes.data, t.shape[0], logits.ctypes.data, hidden.ctypes.data)
        if rc:
            raise ValueError(f"oracle prefill failed ({rc})")
        return logits, hidden

    def extend(self, tokens):
        """More prompt positions after those already in the cache (a prompt run in pieces)."""
        t = _i32(tokens)
        logits = np.empty(self.d["vocab"], np.float32)
        hidden = np.empty(self.d["dim"], np.float32)
        rc = _load().or_extend(self._h, t.ctypes.data, t.shape[0], logits.ctypes.data, hidden.ctypes.data)
        if rc:
            raise ValueError(f"oracle extend failed ({rc})")
        return logits, hidden

    def prefill_chunked(self, tokens, chunk=256):
        """Prefill in pieces of `chunk` positions (the same result as one prefill)."""
        t = _i32(tokens)
        logits, hidden = self.prefill(t[:chunk])
        for a in range(chunk, t.shape[0], chunk):
            logits, hidden = self.extend(t[a:a + chunk])
        return logits, hidden

    def step(self, vals):
        v = _i32(vals)
        logits = np.empty(self.d["vocab"], np.float32)
        hidden = np.empty(self.d["dim"], np.float32)
        rc = _load().or_step(self._h, v.ctypes.data, logits.ctypes.data, hidden.ctypes.data)
        if rc:
            raise ValueError(f"oracle step failed ({rc})")
        return logits, hidden

    def fast_logits(self, hidden, prefix, rows=False):
        h = _f32(hidden)
        p = _i32(prefix)
        k = p.size
        lg = np.empty(self.d["codebook_size"], np.float32)
        rw = np.empty((k + 1, self.d["fast_dim"]), np.float32) if rows else None
        rc = _load().or_fast_forward(self._h, h.ctypes.data, p.ctypes.data, k, lg.ctypes.data,
                                     None if rw is None else rw.ctypes.data)
        if rc:
            raise ValueError(f"oracle fast_forward failed ({rc})")
        return (lg, rw) if rows else lg

    def kv(self, layer, s0, n):
        d = self.d
        k = np.empty((n, d["n_kv_head"], d["head_dim"]), np.float32)
        v = np.empty_like(k)
        if _load().or_kv_io(self._h, layer, s0, n, k.ctypes.data, v.ctypes.data, 0):
            raise ValueError("kv range")
        return k, v

    def set_kv_f16(self, layer, k16, v16):
        """Slots 0..n-1 of one layer from fp16 bit patterns (uint16) in [kv_head][n][head_dim] order."""
        k16 = np.ascontiguousarray(k16, dtype=np.uint16)
        v16 = np.ascontiguousarray(v16, dtype=np.uint16)
        if _load().or_kv_set_f16(self._h, layer, k16.shape[1], k16.ctypes.data, v16.ctypes.data):
            raise ValueError("kv range")

    def head(self, x_last):
        """Final norm + tied logits of a residual: (logits over the vocabulary, normalised hidden)."""
        x = _f32(x_last)
        logits = np.empty(self.d["vocab"], np.float32)
        hidden = np.empty(self.d["dim"], np.float32)
        _load().or_head(self._h, x.ctypes.data, logits.ctypes.data, hidden.ctypes.data)
        return logits, hidden

    def import_state(self, k16, v16, x_last):
        """Stream state without a prompt: K/V fp16 [L][kv_head][n][head_dim] into slots 0..n-1,
        position n, and the head's outputs on x_last (what a prefill of n positions leaves)."""
        n = k16.shape[2]
        for l in range(self.d["n_layer"]):
            self.set_kv_f16(l, k16[l], v16[l])
        self.set_pos(n)
        return self.head(x_last)

    def set_kv(self, layer, s0, k, v):
        k, v = _f32(k), _f32(v)
        if _load().or_kv_io(self._h, layer, s0, k.shape[0], k.ctypes.data, v.ctypes.data, 1):
            raise ValueError("kv range")


# ------------------------------------------------------------ codec front

def codec_latent(quantizers, codes, n_frames):
    """Codec quantizer decode, lookup-and-sum part (ch.02 §3.5: semantic VQ quantizers.0 plus the
    residual VQs quantizers.i, added level by level): latent[f] = Σ_cb Q_cb[codes[cb*n_frames + f]],
    the bf16 codebook rows widened exactly to fp32 and added in codebook order.  The upsampling and
    the waveform decoder that follow on the page are not part of it."""
    out = None
    for cb, q in enumerate(quantizers):
        rows = np.asarray(codes[cb * n_frames:(cb + 1) * n_frames], np.int64)
        widened = (np.asarray(q, np.uint16)[rows].astype(np.uint32) << 16).view(np.float32)
        out = widened.copy() if out is None else (out + widened).astype(np.float32)
    return out


# ------------------------------------------------------------ generation loop

def admissible_ids(d):
    """Token ids left finite by sem_mask, in the order used for admissible-logit vectors:
    sem_begin..sem_end, then im_end."""
    return np.concatenate([np.arange(d["sem_begin"], d["sem_end"] + 1, dtype=np.int32),
                           np.array([d["im_end"]], np.int32)])


def sem_mask(d, block_end: bool):
    """Additive vocabulary mask (ch.06 §5): -inf everywhere, 0 on [sem_begin..sem_end] and on
    im_end; with ``block_end`` (ch.06 §5.3, step < min_tokens_before_end) im_end is -inf too."""
    m = np.full(d["vocab"], -np.inf, np.float32)
    m[d["sem_begin"]:d["sem_end"] + 1] = 0.0
    if not block_end:
        m[d["im_end"]] = 0.0
    return m


def ras_triggered(token, window, d):
    """ch.06 §6: resample when the new main token already sits in the window of recent
    tokens and is a semantic id (im_end never triggers)."""
    return (token in window) and d["sem_begin"] <= token <= d["sem_end"]


def sem_code(token, d):
    """ch.06 §5.1-§5.2: sem_code = main_token - semantic_begin, clamped to [0, codebook_size-1]."""
    return int(min(max(token - d["sem_begin"], 0), d["codebook_size"] - 1))


def compact(frames_codes, d):
    """ch.06 §8: [n_frames][NCB] -> flat codes[cb * n_frames + f]."""
    n = len(frames_codes)
    out = np.zeros(d["n_codebooks"] * n, np.int32)
    for f, cs in enumerate(frames_codes):
        for cb, c in enumerate(cs):
            out[cb * n + f] = c
    return out


N_DRAW_SLOTS = 11   # per-frame draw slots: main, redraw, codebooks 1..9 (unused slots -1)


def run_frames(sess: Session, logits, hidden, n_frames, s, expo, forced=None, window=None, frame0=0,
               trace=True):
    """Frame loop of ch.06 §5.1 from a state (logits, hidden) left by prefill or a step.

    ``s``: sampling dict (temperature, top_p, ras_temperature, ras_top_p, top_k, ras_window,
    min_tokens_before_end).  ``expo``: [n_frames][11][top_k] exponential variates, draw order
    main, redraw, then codebooks 1..9 (Mizuoto page, "parity with upstream").  ``forced``
    (optional [n_frames][11] ints) replaces each draw's outcome, leaving every other rule in place.
    Returns a dict with the emitted frames and, if ``trace``, per-frame logits/diagnostics.
    """
    d = sess.d
    ncb = d["n_codebooks"]
    window = [] if window is None else list(window)
    adm = admissible_ids(d)
    out = dict(codes=[], draws=[], diags=[], main_logits=[], hidden=[], fast_logits=[], tokens=[],
               stopped=False, window=None)
    for fi in range(n_frames):
        f = frame0 + fi
        lp = logits + sem_mask(d, f < s["min_tokens_before_end"])
        e = expo[fi]
        draws, diags = [], []
        d0, g0 = draw(lp, s["temperature"], s["top_p"], s["top_k"], e[0])
        if trace:
            out["main_logits"].append(logits[adm].copy())
            out["hidden"].append(hidden.copy())
        draws.append(d0)
        diags.append(g0)
        if forced is not None:
            d0 = int(forced[fi][0])
        if d0 == d["im_end"]:
            out["stopped"] = True
            out["draws"].append(draws + [-1] * (N_DRAW_SLOTS - len(draws)))
            out["diags"].append(diags)
            break
        d1, g1 = draw(lp, s["ras_temperature"], s["ras_top_p"], s["top_k"], e[1])
        draws.append(d1)
        diags.append(g1)
        if forced is not None:
            d1 = int(forced[fi][1])
        token = d1 if ras_triggered(d0, window, d) else d0
        codes = [sem_code(token, d)]
        fl_all = []
        for c in range(1, ncb):
            fl = sess.fast_logits(hidden, codes)
            dc, gc = draw(fl, s["temperature"], s["top_p"], s["top_k"], e[1 + c])
            draws.append(dc)
            diags.append(gc)
            if forced is not None:
                dc = int(forced[fi][1 + c])
            codes.append(dc)
            if trace:
                fl_all.append(fl)
        out["codes"].append(codes)
        out["tokens"].append(token)
        out["draws"].append(draws + [-1] * (N_DRAW_SLOTS - len(draws)))
        out["diags"].append(diags)
        if trace:
            out["fast_logits"].append(np.stack(fl_all))
        window.append(token)
        if len(window) > s["ras_window"]:
            window.pop(0)
        logits, hidden = sess.step([token] + codes)
    out["window"] = window
    out["logits"], out["last_hidden"] = logits, hidden
    out["flat"] = compact(out["codes"], d)
    return out


def generate(sess: Session, prompt, n_frames, s, expo, forced=None, trace=True):
    """prefill + frame loop (ch.06 §5.1); returns run_frames' dict plus the prefill outputs."""
    logits, hidden = sess.prefill(prompt)
    res = run_frames(sess, logits, hidden, n_frames, s, expo, forced=forced, trace=trace)
    res["prefill_logits"], res["prefill_hidden"] = logits, hidden
    return res
