"""Seeded synthetic inputs for the S2-Pro Dual-AR frame decode.

Holds no arithmetic of the method: only the model shapes of the five workloads,
the weight-table order (an interface both sides agree on) and counter-based
random numbers (SplitMix64; see ``synth.c``).  Both the CPU oracle and the CUDA
path are fed from here.  The weights, prompts and exponential variates are
synthetic stand-ins for trained S2-Pro weights and real prompts, which these
runs do not have.

Workloads (shapes from the s2cpp-analysis pages, ch.02 "Architecture & data flow"
§2 dims table and ch.04 "Model loading & GGUF" §2.2 hyper-parameters):

* ``tiny``      — tiny Dual-AR in fp32 (the small case the oracle finishes in seconds)
* ``fast``      — Fast-AR alone at S2-Pro shapes, bf16, teacher-forced windows
* ``frame``     — full frame decode at S2-Pro shapes, bf16, batch 1
* ``serving``   — 32 independent streams, prompts of 512..4096 positions
* ``longctx``   — 8 streams × 30000 prompt positions into 32768 KV slots
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading
import zlib

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libs2synth.so")
_lib = None
_lock = threading.Lock()

# dtype codes shared by the dims dicts below
F32, BF16, F16 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile ``synth.c`` into ``libs2synth.so`` next to it (plain gcc, OpenMP)."""
    src = os.path.join(_HERE, "synth.c")
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(src):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                               "-std=c11", src, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            u64, i64, i32, dbl, vp = (ctypes.c_uint64, ctypes.c_int64, ctypes.c_int32,
                                      ctypes.c_double, ctypes.c_void_p)
            lib.synth_normal_f32.argtypes = [u64, u64, i64, dbl, dbl, vp]
            lib.synth_normal_bf16.argtypes = [u64, u64, i64, dbl, dbl, vp]
            lib.synth_normal_f16.argtypes = [u64, u64, i64, dbl, dbl, vp]
            lib.synth_exponential_f32.argtypes = [u64, u64, i64, vp]
            lib.synth_uniform_f64.argtypes = [u64, u64, i64, vp]
            lib.synth_uniform_int.argtypes = [u64, u64, i64, i32, i32, vp]
            for f in (lib.synth_normal_f32, lib.synth_normal_bf16, lib.synth_normal_f16, lib.synth_exponential_f32,
                      lib.synth_uniform_f64, lib.synth_uniform_int):
                f.restype = None
            _lib = lib
    return _lib


# ---------------------------------------------------------------------------
# raw generators
# ---------------------------------------------------------------------------

def normal_f32(seed: int, stream: int, n: int, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    out = np.empty(n, np.float32)
    _load().synth_normal_f32(seed, stream, n, mean, std, out.ctypes.data)
    return out


def normal_bf16(seed: int, stream: int, n: int, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    """bf16 bit patterns (uint16)."""
    out = np.empty(n, np.uint16)
    _load().synth_normal_bf16(seed, stream, n, mean, std, out.ctypes.data)
    return out


def normal_f16(seed: int, stream: int, n: int, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    """fp16 bit patterns (uint16)."""
    out = np.empty(n, np.uint16)
    _load().synth_normal_f16(seed, stream, n, mean, std, out.ctypes.data)
    return out


def exponential_f32(seed: int, stream: int, n: int) -> np.ndarray:
    out = np.empty(n, np.float32)
    _load().synth_exponential_f32(seed, stream, n, out.ctypes.data)
    return out


def uniform_f64(seed: int, stream: int, n: int) -> np.ndarray:
    out = np.empty(n, np.float64)
    _load().synth_uniform_f64(seed, stream, n, out.ctypes.data)
    return out


def uniform_int(seed: int, stream: int, n: int, lo: int, hi: int) -> np.ndarray:
    out = np.empty(n, np.int32)
    _load().synth_uniform_int(seed, stream, n, lo, hi, out.ctypes.data)
    return out


def bf16_to_f32(u16: np.ndarray) -> np.ndarray:
    return (u16.astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------------------
# model shapes
# ---------------------------------------------------------------------------

_S2PRO = dict(
    dim=2560, n_layer=36, n_head=32, n_kv_head=8, head_dim=128, ffn=9728, vocab=155776,
    sem_begin=151678, sem_end=155773, im_end=151645, n_codebooks=10, codebook_size=4096,
    sem_scale=1.0 / math.sqrt(11.0), norm_eps=1e-6, rope_base=1e6, qk_norm=1, rope_table_bf16=1,
    fast_dim=2560, fast_n_layer=4, fast_n_head=32, fast_n_kv_head=8, fast_head_dim=128,
    fast_ffn=9728, fast_window=11, has_fast_project_in=1,
    weight_dtype=BF16, kv_dtype=F16, weight_fp8=0,
)

_TINY = dict(
    dim=256, n_layer=4, n_head=4, n_kv_head=2, head_dim=64, ffn=768, vocab=4608,
    sem_begin=4096, sem_end=4159, im_end=4160, n_codebooks=4, codebook_size=64,
    sem_scale=1.0 / math.sqrt(5.0), norm_eps=1e-6, rope_base=1e6, qk_norm=1, rope_table_bf16=1,
    fast_dim=256, fast_n_layer=2, fast_n_head=4, fast_n_kv_head=2, fast_head_dim=64,
    fast_ffn=768, fast_window=5, has_fast_project_in=1,
    weight_dtype=F32, kv_dtype=F32, weight_fp8=0,
)

_SAMPLING = dict(temperature=0.8, top_p=0.8, ras_temperature=1.0, ras_top_p=0.9, top_k=30, ras_window=10)

#: workload table; ``streams``/``prompt``/``frames`` describe the synthetic inputs
CONFIGS = {
    "tiny": dict(dims=_TINY, streams=1, frames=16, min_tokens=16, kv_slots=64,
                 weight_seed=0, input_seed=0),
    "fast": dict(dims=dict(_S2PRO, n_layer=0), streams=1, frames=1000, min_tokens=0, kv_slots=0,
                 weight_seed=0, input_seed=1),
    "frame": dict(dims=_S2PRO, streams=1, frames=256, min_tokens=32, kv_slots=32768,
                  weight_seed=0, input_seed=2),
    "serving": dict(dims=_S2PRO, streams=32, frames=128, min_tokens=128, kv_slots=4224,
                    weight_seed=0, input_seed=3),
    "longctx": dict(dims=_S2PRO, streams=8, frames=256, min_tokens=256, kv_slots=32768,
                    weight_seed=0, input_seed=4),
}


def sampling(cfg: str, **over) -> dict:
    s = dict(_SAMPLING, min_tokens_before_end=CONFIGS[cfg]["min_tokens"], max_frames=CONFIGS[cfg]["frames"])
    s.update(over)
    return s


# ---------------------------------------------------------------------------
# weight table (fixed name order; an interface, not arithmetic)
# ---------------------------------------------------------------------------

_LAYER_NAMES = ("attention_norm", "attention.wqkv", "attention.q_norm", "attention.k_norm",
                "attention.wo", "ffn_norm", "feed_forward.w1", "feed_forward.w3", "feed_forward.w2")


def _layer_shapes(dim, nh, nkv, hd, ffn):
    return [(dim,), ((nh + 2 * nkv) * hd, dim), (hd,), (hd,), (dim, nh * hd), (dim,),
            (ffn, dim), (ffn, dim), (dim, ffn)]


def weight_specs(d: dict):
    """List of (name, shape, is_norm) in the weight-table order.

    Order: embeddings, codebook_embeddings, norm, then 9 tensors per Slow-AR layer
    (attention_norm, attention.wqkv, attention.q_norm, attention.k_norm, attention.wo,
    ffn_norm, feed_forward.w1, feed_forward.w3, feed_forward.w2), then fast_project_in,
    fast_embeddings, fast_norm, fast_output, then the same 9 per Fast-AR layer.
    Tensor names follow the GGUF names on ch.04 "Model loading & GGUF" §3.
    """
    D, ncb, cbs = d["dim"], d["n_codebooks"], d["codebook_size"]
    specs = [("embeddings", (d["vocab"], D), False),
             ("codebook_embeddings", (ncb * cbs, D), False),
             ("norm", (D,), True)]
    for i in range(d["n_layer"]):
        for nm, shp in zip(_LAYER_NAMES, _layer_shapes(D, d["n_head"], d["n_kv_head"], d["head_dim"], d["ffn"])):
            specs.append((f"layers.{i}.{nm}", shp, nm.endswith("norm")))
    Df = d["fast_dim"]
    specs += [("fast_project_in", (Df, D), False), ("fast_embeddings", (cbs, Df), False),
              ("fast_norm", (Df,), True), ("fast_output", (cbs, Df), False)]
    for i in range(d["fast_n_layer"]):
        for nm, shp in zip(_LAYER_NAMES, _layer_shapes(Df, d["fast_n_head"], d["fast_n_kv_head"],
                                                       d["fast_head_dim"], d["fast_ffn"])):
            specs.append((f"fast_layers.{i}.{nm}", shp, nm.endswith("norm")))
    return specs


def make_weights(d: dict, seed: int = 0, std: float = 0.02, norm_jitter: float = 0.0,
                 skip_slow: bool | None = None):
    """Synthetic weights in table order.  Matrices ~ N(0, std); norm weights 1 (+ N(0, norm_jitter)).

    Returns a list of numpy arrays: float32 for fp32 models, uint16 bf16 patterns for bf16
    models.  With ``skip_slow`` (default: when the model has no Slow-AR layers) the
    embeddings / codebook_embeddings / norm entries are None.
    """
    if skip_slow is None:
        skip_slow = d["n_layer"] == 0
    out = []
    for name, shape, is_norm in weight_specs(d):
        idx = tensor_stream(name)
        if skip_slow and name in ("embeddings", "codebook_embeddings", "norm"):
            out.append(None)
            continue
        if name == "fast_project_in" and not d["has_fast_project_in"]:
            out.append(None)
            continue
        n = int(np.prod(shape))
        mean, s = (1.0, norm_jitter) if is_norm else (0.0, std)
        if d["weight_dtype"] == BF16:
            arr = normal_bf16(seed, idx, n, mean, s) if s > 0 else _const_bf16(n, mean)
        else:
            arr = normal_f32(seed, idx, n, mean, s) if s > 0 else np.full(n, mean, np.float32)
        out.append(arr.reshape(shape))
    return out


def tensor_stream(name: str) -> int:
    """Generator stream of a weight tensor, keyed by its name (so a tensor has the same values in
    every workload that contains it, e.g. the Fast-AR weights of the full model and of the
    Fast-AR-alone workload)."""
    return zlib.crc32(name.encode())


def _const_bf16(n, v):
    return np.full(n, np.float32(v)).view(np.uint32).__rshift__(16).astype(np.uint16)


# ---------------------------------------------------------------------------
# prompts and random draws
# ---------------------------------------------------------------------------

def _prompt(d, seed, stream, n_text, n_ref):
    """(n_text + n_ref) x (NCB+1) int32, column-major token layout [t][row].

    Row 0: uniform text ids in [0, sem_begin) then uniform semantic ids in [sem_begin, sem_end];
    rows 1..NCB: uniform codes in [0, codebook_size) at reference positions, 0 at text positions
    (ch.02 "Architecture & data flow" §3.1).
    """
    ncb, T = d["n_codebooks"], n_text + n_ref
    base = 1_000_000 + 64 * stream
    p = np.zeros((T, ncb + 1), np.int32)
    p[:n_text, 0] = uniform_int(seed, base + 0, n_text, 0, d["sem_begin"] - 1)
    p[n_text:, 0] = uniform_int(seed, base + 1, n_ref, d["sem_begin"], d["sem_end"])
    codes = uniform_int(seed, base + 2, n_ref * ncb, 0, d["codebook_size"] - 1).reshape(n_ref, ncb)
    p[n_text:, 1:] = codes
    return p


def make_prompt(d: dict, seed: int, stream: int, n_text: int, n_ref: int) -> np.ndarray:
    """A prompt of the given text / reference split for any model shape (same recipe as the
    workloads' prompts)."""
    return _prompt(d, seed, stream, n_text, n_ref)


#: a small bf16 model with four query heads per KV head (the grouping of S2-Pro), for quick
#: checks of the batched decode path
MINI = dict(_TINY, n_head=4, n_kv_head=1, ffn=512, fast_n_head=4, fast_n_kv_head=1, fast_ffn=512,
            weight_dtype=BF16, kv_dtype=F16)


def prompt_lengths(cfg: str):
    c = CONFIGS[cfg]
    if cfg == "tiny":
        return [32]
    if cfg == "frame":
        return [512]
    if cfg == "serving":
        return [int(uniform_int(c["input_seed"] + i, 7, 1, 512, 4096)[0]) for i in range(c["streams"])]
    if cfg == "longctx":
        return [30000] * c["streams"]
    raise ValueError(cfg)


def prompt(cfg: str, stream: int = 0, length: int | None = None) -> np.ndarray:
    """Prompt matrix of one stream of a workload, [T][NCB+1] int32."""
    c = CONFIGS[cfg]
    d = c["dims"]
    if cfg == "tiny":
        return _prompt(d, c["input_seed"], stream, 24, 8)
    if cfg == "frame":
        L = length or 512
        n_text = (L * 3) // 4
        return _prompt(d, c["input_seed"], stream, n_text, L - n_text)
    if cfg == "serving":
        L = length or prompt_lengths(cfg)[stream]
        n_text = int(round(0.75 * L))
        return _prompt(d, c["input_seed"] + stream, stream, n_text, L - n_text)
    if cfg == "longctx":
        L = length or 30000
        n_text = min(1000, L // 30)
        return _prompt(d, c["input_seed"] + stream, stream, n_text, L - n_text)
    raise ValueError(cfg)


N_DRAWS = 11      # per frame: main, repetition-aware redraw, 9 Fast-AR codebooks
TOP_K = 30


def expo(seed: int, stream: int, n_frames: int, first_frame: int = 0) -> np.ndarray:
    """Exponential variates for the sampler, [n_frames][11][30] fp32.

    Index [f][draw][rank]: frame f, draw 0 = main token, 1 = repetition-aware redraw,
    2..10 = Fast-AR codebooks 1..9; rank within the top-30 candidates.
    """
    per = N_DRAWS * TOP_K
    full = exponential_f32(seed, 2_000_000 + stream, (first_frame + n_frames) * per)
    return full[first_frame * per:].reshape(n_frames, N_DRAWS, TOP_K)


def kv_state(seed: int, stream: int, d: dict, n_pos: int):
    """Synthetic decode state of one stream, standing in for a prefilled prompt of n_pos positions
    (used where an fp32 CPU prefill of the prompt would take too long).

    K and V ~ N(0, 1) as fp16 bit patterns [n_layer][n_kv_head][n_pos][head_dim] (the scale of
    normalised keys and of values projected from a normalised residual with N(0, 0.02) weights),
    and the last residual x ~ N(0, 1) fp32 [dim].  Values of (layer, head) come from their own
    generator stream indexed by slot * head_dim + element, so a shorter state is a prefix of a
    longer one under the same seed and stream.
    """
    L, H, hd = d["n_layer"], d["n_kv_head"], d["head_dim"]
    base = 4_000_000 + 4096 * stream
    k = np.empty((L, H, n_pos, hd), np.uint16)
    v = np.empty_like(k)
    for l in range(L):
        for g in range(H):
            j = 2 * (l * H + g)
            k[l, g] = normal_f16(seed, base + j, n_pos * hd).reshape(n_pos, hd)
            v[l, g] = normal_f16(seed, base + j + 1, n_pos * hd).reshape(n_pos, hd)
    x = normal_f32(seed, base + 4095, d["dim"])
    return k, v, x


#: codec quantizer shape (the pages give none): one codebook per code row, 1024-wide latent
CODEC_DIM = 1024


def codec_quantizers(seed: int, n_codebooks: int, codebook_size: int, dim: int = CODEC_DIM):
    """Synthetic codec VQ codebooks (semantic, then residual), bf16 N(0, 1) [codebook_size][dim]."""
    return [normal_bf16(seed, 6_000_000 + cb, codebook_size * dim).reshape(codebook_size, dim)
            for cb in range(n_codebooks)]


def fast_inputs(seed: int, n_frames: int, d: dict):
    """Fast-AR-alone inputs: hidden ~ N(0,1)^D per frame, prefix codes uniform in [0, CBS)."""
    hid = normal_f32(seed, 3_000_000, n_frames * d["dim"]).reshape(n_frames, d["dim"])
    codes = uniform_int(seed, 3_000_001, n_frames * (d["n_codebooks"] - 1), 0,
                        d["codebook_size"] - 1).reshape(n_frames, d["n_codebooks"] - 1)
    return hid, codes
