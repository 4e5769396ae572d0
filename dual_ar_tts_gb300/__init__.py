"""GB300 (sm_103a) Dual-AR frame decoder for S2-Pro — thin Python binding of ``libs2frame.so``.

The functions named ``s2_*`` mirror the C ABI in ``include/s2frame.h`` one to one and only
marshal arguments; every step of the decode runs in the library's CUDA kernels.  PyTorch is
used for device memory and streams.  There is no CPU fallback: if the CUDA library is missing
or no GPU is present, calls raise.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libs2frame.so")

S2_F32, S2_BF16, S2_F16 = 0, 1, 2
S2_OK, S2_EINVAL, S2_ENOMEM, S2_ECAPACITY, S2_ECUDA, S2_ETIMEOUT, S2_ESTATE = range(7)
STATUS_NAMES = {0: "S2_OK", 1: "S2_EINVAL", 2: "S2_ENOMEM", 3: "S2_ECAPACITY", 4: "S2_ECUDA", 5: "S2_ETIMEOUT",
                6: "S2_ESTATE"}

EXPORTS = ("s2_weight_count", "s2_weight_info", "s2_frame_workspace_bytes", "s2_frame_init", "s2_prefill",
           "s2_decode_frames", "s2_fast_logits", "s2_sync_status", "s2_set_spin_limit", "s2_set_trace",
           "s2_phase_count", "s2_frame_free", "s2_last_error", "s2_fast_logits_static", "s2_stream_import",
           "s2_stop_stream", "s2_stream_progress", "s2_codec_latent", "s2_quantize_e4m3", "s2_set_barrier_base",
           "s2_draw")


class s2_dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("dim", "n_layer", "n_head", "n_kv_head", "head_dim", "ffn", "vocab",
                                            "sem_begin", "sem_end", "im_end", "n_codebooks", "codebook_size")] + \
               [(n, ctypes.c_float) for n in ("sem_scale", "norm_eps", "rope_base")] + \
               [(n, ctypes.c_int) for n in ("qk_norm", "rope_table_bf16", "fast_dim", "fast_n_layer", "fast_n_head",
                                            "fast_n_kv_head", "fast_head_dim", "fast_ffn", "fast_window",
                                            "has_fast_project_in", "weight_dtype", "kv_dtype", "weight_fp8")]


class s2_sampling(ctypes.Structure):
    _fields_ = [("temperature", ctypes.c_float), ("top_p", ctypes.c_float), ("ras_temperature", ctypes.c_float),
                ("ras_top_p", ctypes.c_float), ("top_k", ctypes.c_int), ("ras_window", ctypes.c_int),
                ("min_tokens_before_end", ctypes.c_int), ("max_frames", ctypes.c_int)]


class s2_debug_taps(ctypes.Structure):
    _fields_ = [("main_logits", ctypes.c_void_p), ("fast_logits", ctypes.c_void_p), ("hidden", ctypes.c_void_p),
                ("draws", ctypes.c_void_p)]


class S2Error(RuntimeError):
    def __init__(self, fn, code, msg):
        super().__init__(f"{fn} -> {STATUS_NAMES.get(code, code)}: {msg}")
        self.code = code


_lib = None


def load(path: str = LIB_PATH):
    """Load the CUDA library (build it first with ``dual_ar_tts_gb300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: run `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(path)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong, ctypes.c_size_t
    P = ctypes.POINTER
    sig = {
        "s2_weight_count": (i32, [P(s2_dims)]),
        "s2_weight_info": (i64, [P(s2_dims), i32, ctypes.c_char_p, i32]),
        "s2_frame_workspace_bytes": (sz, [P(s2_dims), i32, i32]),
        "s2_frame_init": (i32, [P(s2_dims), P(vp), i32, vp, sz, i32, i32, P(vp)]),
        "s2_prefill": (i32, [vp, i32, P(i32), vp, P(i32), vp]),
        "s2_decode_frames": (i32, [vp, i32, P(i32), i32, P(s2_sampling), vp, vp, vp, vp, P(s2_debug_taps), vp]),
        "s2_fast_logits": (i32, [vp, i32, vp, vp, vp, vp]),
        "s2_sync_status": (i32, [vp, vp]),
        "s2_set_spin_limit": (i32, [vp, i64]),
        "s2_set_trace": (i32, [vp, vp, i32]),
        "s2_set_barrier_base": (i32, [vp, ctypes.c_uint]),
        "s2_phase_count": (i32, [vp, i32]),
        "s2_frame_free": (i32, [vp]),
        "s2_last_error": (ctypes.c_char_p, [vp]),
        "s2_fast_logits_static": (i32, [P(s2_dims), P(vp), i32, i32, vp, vp, vp, vp, vp]),
        "s2_stream_import": (i32, [vp, i32, i32, vp, vp, vp, vp]),
        "s2_stop_stream": (i32, [vp, i32, vp]),
        "s2_codec_latent": (i32, [i32, i32, i32, P(vp), i32, vp, vp, vp, vp]),
        "s2_quantize_e4m3": (i32, [vp, ctypes.c_longlong, i32, vp, vp, vp]),
        "s2_stream_progress": (i32, [vp, i32, P(i32), vp, vp]),
        "s2_draw": (i32, [i32, vp, i32, i32, i32, i32, ctypes.c_float, ctypes.c_float, vp, vp, vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(fn, rc, ctx=None):
    if rc != S2_OK:
        raise S2Error(fn, rc, load().s2_last_error(ctx).decode())
    return rc


def _ints(seq):
    arr = (ctypes.c_int * len(seq))(*[int(v) for v in seq])
    return arr


# ------------------------------------------------------------------ the C ABI

def make_dims(d: dict) -> s2_dims:
    s = s2_dims()
    for name, _ in s2_dims._fields_:
        setattr(s, name, d.get(name, 0) if name == "weight_fp8" else d[name])
    return s


def s2_weight_count(dims: s2_dims) -> int:
    return load().s2_weight_count(ctypes.byref(dims))


def s2_weight_info(dims: s2_dims, i: int):
    buf = ctypes.create_string_buffer(128)
    n = load().s2_weight_info(ctypes.byref(dims), i, buf, 128)
    return buf.value.decode(), n


def s2_frame_workspace_bytes(dims: s2_dims, max_streams: int, kv_slots: int) -> int:
    return load().s2_frame_workspace_bytes(ctypes.byref(dims), max_streams, kv_slots)


def s2_frame_init(dims: s2_dims, weight_ptrs, workspace_ptr: int, ws_bytes: int, max_streams: int, kv_slots: int):
    n = len(weight_ptrs)
    arr = (ctypes.c_void_p * n)(*[p if p else None for p in weight_ptrs])
    out = ctypes.c_void_p()
    rc = load().s2_frame_init(ctypes.byref(dims), arr, n, workspace_ptr, ws_bytes, max_streams, kv_slots,
                              ctypes.byref(out))
    _check("s2_frame_init", rc, None)
    return out.value


def s2_prefill(ctx, stream_ids, tokens_ptr: int, lengths, stream: int = 0):
    rc = load().s2_prefill(ctx, len(stream_ids), _ints(stream_ids), tokens_ptr, _ints(lengths), stream)
    return _check("s2_prefill", rc, ctx)


def s2_stream_import(ctx, stream_id: int, n_pos: int, k_ptr: int, v_ptr: int, x_last_ptr: int, stream: int = 0):
    rc = load().s2_stream_import(ctx, stream_id, n_pos, k_ptr, v_ptr, x_last_ptr, stream)
    return _check("s2_stream_import", rc, ctx)


def s2_stop_stream(ctx, stream_id: int, side_stream: int = 0):
    return _check("s2_stop_stream", load().s2_stop_stream(ctx, stream_id, side_stream), ctx)


def s2_stream_progress(ctx, stream_ids, out_ptr: int, side_stream: int = 0):
    rc = load().s2_stream_progress(ctx, len(stream_ids), _ints(stream_ids), out_ptr, side_stream)
    return _check("s2_stream_progress", rc, ctx)


def s2_codec_latent(n_codebooks: int, codebook_size: int, dim: int, quantizer_ptrs, n_frames: int, codes_ptr: int,
                    latent_ptr: int, status_ptr: int | None = None, stream: int = 0):
    """Codec latent = Σ_cb quantizer_cb[code] per frame (device pointers; see s2frame.h)."""
    arr = (ctypes.c_void_p * len(quantizer_ptrs))(*quantizer_ptrs)
    rc = load().s2_codec_latent(n_codebooks, codebook_size, dim, arr, n_frames, codes_ptr, latent_ptr, status_ptr,
                                stream)
    return _check("s2_codec_latent", rc)


def s2_quantize_e4m3(w_ptr: int, rows: int, cols: int, codes_ptr: int, scales_ptr: int, stream: int = 0):
    """e4m3 codes + fp32 row scales of bf16 rows (device pointers; see s2frame.h)."""
    return _check("s2_quantize_e4m3", load().s2_quantize_e4m3(w_ptr, rows, cols, codes_ptr, scales_ptr, stream))


def s2_draw(rows: int, logits_ptr: int, n: int, sem_begin: int, im_end: int, block_end: bool, temperature: float,
            top_p: float, expo_ptr: int, out_ptr: int, stream: int = 0):
    """The S2 draw on device logits rows (see s2frame.h)."""
    rc = load().s2_draw(rows, logits_ptr, n, sem_begin, im_end, 1 if block_end else 0, temperature, top_p, expo_ptr,
                        out_ptr, stream)
    return _check("s2_draw", rc)


def draw(logits, expo, temperature: float, top_p: float, sem_begin: int = -1, im_end: int = 0,
         block_end: bool = False):
    """Device fp32 logits [rows][n] and variates [rows][30] (torch) -> drawn ids, int32 [rows]."""
    import torch
    if logits.dtype != torch.float32 or logits.dim() != 2 or not logits.is_cuda:
        raise ValueError("draw takes 2-D fp32 CUDA logits")
    if expo.dtype != torch.float32 or tuple(expo.shape) != (logits.shape[0], 30) or not expo.is_cuda:
        raise ValueError("draw takes fp32 CUDA variates of shape [rows][30]")
    logits, expo = logits.contiguous(), expo.contiguous()
    out = torch.empty(logits.shape[0], dtype=torch.int32, device=logits.device)
    s2_draw(logits.shape[0], logits.data_ptr(), logits.shape[1], sem_begin, im_end, block_end, temperature, top_p,
            expo.data_ptr(), out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    return out


def quantize_e4m3(w):
    """Device bf16 matrix (torch, [rows][cols]) -> (uint8 codes [rows][cols], fp32 scales [rows])."""
    import torch
    if w.dtype != torch.bfloat16 or w.dim() != 2 or not w.is_cuda:
        raise ValueError("quantize_e4m3 takes a 2-D bf16 CUDA tensor")
    w = w.contiguous()
    codes = torch.empty(w.shape, dtype=torch.uint8, device=w.device)
    scales = torch.empty(w.shape[0], dtype=torch.float32, device=w.device)
    s2_quantize_e4m3(w.data_ptr(), w.shape[0], w.shape[1], codes.data_ptr(), scales.data_ptr(),
                     torch.cuda.current_stream().cuda_stream)
    return codes, scales


def s2_decode_frames(ctx, stream_ids, n_frames: int, params, expo_ptr: int, forced_ptr: int | None, codes_ptr: int,
                     n_out_ptr: int, taps: s2_debug_taps | None = None, stream: int = 0):
    n = len(stream_ids)
    arr = (s2_sampling * n)(*params)
    rc = load().s2_decode_frames(ctx, n, _ints(stream_ids), n_frames, arr, expo_ptr, forced_ptr, codes_ptr, n_out_ptr,
                                 ctypes.byref(taps) if taps is not None else None, stream)
    return _check("s2_decode_frames", rc, ctx)


def s2_fast_logits(ctx, n_frames: int, hidden_ptr: int, prefix_ptr: int, logits_ptr: int, stream: int = 0):
    rc = load().s2_fast_logits(ctx, n_frames, hidden_ptr, prefix_ptr, logits_ptr, stream)
    return _check("s2_fast_logits", rc, ctx)


def s2_sync_status(ctx, stream: int = 0) -> int:
    return load().s2_sync_status(ctx, stream)


def s2_set_spin_limit(ctx, limit: int):
    return _check("s2_set_spin_limit", load().s2_set_spin_limit(ctx, limit), ctx)


def s2_set_barrier_base(ctx, base: int):
    return _check("s2_set_barrier_base", load().s2_set_barrier_base(ctx, base), ctx)


def s2_set_trace(ctx, buf_ptr: int | None, capacity: int):
    return _check("s2_set_trace", load().s2_set_trace(ctx, buf_ptr, capacity), ctx)


def s2_phase_count(ctx, fast_only: bool = False) -> int:
    return load().s2_phase_count(ctx, int(bool(fast_only)))


def s2_frame_free(ctx):
    return load().s2_frame_free(ctx)


def s2_last_error(ctx=None) -> str:
    return load().s2_last_error(ctx).decode()


def s2_fast_logits_static(dims: s2_dims, weight_ptrs, n_frames: int, hidden_ptr: int, prefix_ptr: int,
                          logits_ptr: int, status_ptr: int | None = None, stream: int = 0):
    """Fast-AR alone on the library's static scratch: no context, no workspace, no allocation.
    The caller passes every input and output (device pointers)."""
    arr = (ctypes.c_void_p * len(weight_ptrs))(*[p if p else None for p in weight_ptrs])
    rc = load().s2_fast_logits_static(ctypes.byref(dims), arr, len(weight_ptrs), n_frames, hidden_ptr, prefix_ptr,
                                      logits_ptr, status_ptr, stream)
    return _check("s2_fast_logits_static", rc)


def make_sampling(s: dict) -> s2_sampling:
    return s2_sampling(s["temperature"], s["top_p"], s["ras_temperature"], s["ras_top_p"], s["top_k"],
                       s["ras_window"], s["min_tokens_before_end"], s.get("max_frames", 0))


# ------------------------------------------------------- memory-owning helper

class Decoder:
    """Owns the device workspace (a torch tensor) and the weight tensors for one context."""

    def __init__(self, d: dict, weights, max_streams: int = 1, kv_slots: int = 0, device: str = "cuda"):
        import torch
        if not torch.cuda.is_available():
            raise RuntimeError("the frame decoder needs a CUDA GPU")
        load()
        self.d = d
        self.dims = make_dims(d)
        self.weights = weights          # torch device tensors (or None), table order
        ptrs = [w.data_ptr() if w is not None else 0 for w in weights]
        nbytes = s2_frame_workspace_bytes(self.dims, max_streams, kv_slots)
        if nbytes == 0:
            raise S2Error("s2_frame_workspace_bytes", S2_EINVAL, s2_last_error(None))
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=device)
        self.ctx = s2_frame_init(self.dims, ptrs, self.workspace.data_ptr(), nbytes, max_streams, kv_slots)
        self.max_streams = max_streams
        self.kv_slots = kv_slots

    def close(self):
        if getattr(self, "ctx", None):
            s2_frame_free(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def stream(self):
        import torch
        return torch.cuda.current_stream().cuda_stream

    def prefill(self, prompts, stream_ids=None):
        """prompts: list of [T][NCB+1] int32 arrays/tensors (host or device)."""
        import torch
        ids = list(range(len(prompts))) if stream_ids is None else list(stream_ids)
        toks = torch.cat([torch.as_tensor(p, dtype=torch.int32).reshape(-1) for p in prompts]).cuda()
        lens = [int(torch.as_tensor(p).shape[0]) for p in prompts]
        s2_prefill(self.ctx, ids, toks.data_ptr(), lens, self.stream())
        self._keep = toks
        return toks

    def stop(self, stream_id, side_stream=None):
        """Ask a stream to stop at its next frame boundary (takes effect during a running decode
        when side_stream is a non-blocking stream other than the decode's)."""
        import torch
        side = side_stream if side_stream is not None else torch.cuda.Stream()
        s2_stop_stream(self.ctx, stream_id, side.cuda_stream)
        side.synchronize()

    def progress(self, stream_ids, side_stream=None):
        """Frames emitted so far by the running (or last) decode call, per stream id."""
        import numpy as np
        import torch
        side = side_stream if side_stream is not None else torch.cuda.Stream()
        out = np.zeros(len(stream_ids), np.int32)
        s2_stream_progress(self.ctx, list(stream_ids), out.ctypes.data, side.cuda_stream)
        side.synchronize()
        return out

    def import_stream(self, stream_id, k, v, x_last):
        """k, v: device tensors [n_layer][n_kv_head][n_pos][head_dim] of the KV dtype; x_last: [dim] fp32."""
        n_pos = int(k.shape[2])
        s2_stream_import(self.ctx, stream_id, n_pos, k.data_ptr(), v.data_ptr(), x_last.data_ptr(), self.stream())

    def decode(self, n_frames, sampling, expo, forced=None, stream_ids=None, taps=False):
        """expo: [n][n_frames][11][30] float32 (device tensor); forced: optional [n][n_frames][11] int32.
        Returns dict of device tensors (codes, n_out and, with taps, the debug outputs)."""
        import torch
        n = expo.shape[0]
        ids = list(range(n)) if stream_ids is None else list(stream_ids)
        d = self.d
        dev = expo.device
        codes = torch.zeros((n, d["n_codebooks"] * n_frames), dtype=torch.int32, device=dev)
        n_out = torch.zeros(n, dtype=torch.int32, device=dev)
        out = dict(codes=codes, n_out=n_out)
        t = None
        if taps:
            A = d["codebook_size"] + 1
            out["main_logits"] = torch.full((n, n_frames, A), float("nan"), device=dev)
            out["fast_logits"] = torch.full((n, n_frames, d["n_codebooks"] - 1, d["codebook_size"]), float("nan"),
                                            device=dev)
            out["hidden"] = torch.full((n, n_frames, d["dim"]), float("nan"), device=dev)
            out["draws"] = torch.full((n, n_frames, 11), -2, dtype=torch.int32, device=dev)
            t = s2_debug_taps(out["main_logits"].data_ptr(), out["fast_logits"].data_ptr(), out["hidden"].data_ptr(),
                              out["draws"].data_ptr())
        params = [make_sampling(sampling) for _ in range(n)] if isinstance(sampling, dict) else \
            [make_sampling(s) for s in sampling]
        s2_decode_frames(self.ctx, ids, n_frames, params, expo.data_ptr(),
                         forced.data_ptr() if forced is not None else None, codes.data_ptr(), n_out.data_ptr(), t,
                         self.stream())
        return out

    def fast_logits(self, hidden, prefix):
        import torch
        n = hidden.shape[0]
        d = self.d
        out = torch.empty((n, d["n_codebooks"] - 1, d["codebook_size"]), dtype=torch.float32, device=hidden.device)
        s2_fast_logits(self.ctx, n, hidden.data_ptr(), prefix.data_ptr(), out.data_ptr(), self.stream())
        return out

    def sync_status(self) -> int:
        return s2_sync_status(self.ctx, self.stream())


def upload_weights(host_weights, device="cuda"):
    """Host arrays (fp32, or uint16 bf16 patterns) -> torch device tensors (bf16 / fp32)."""
    import numpy as np
    import torch
    out = []
    for w in host_weights:
        if w is None:
            out.append(None)
            continue
        if w.dtype == np.uint16:
            t = torch.from_numpy(w.view(np.int16)).to(device).view(torch.bfloat16)
        else:
            t = torch.from_numpy(np.ascontiguousarray(w, dtype=np.float32)).to(device)
        out.append(t)
    return out


def serve(decoder, requests, slots, frames_per_call, sampling, expo_fn, forced_fn=None):
    """Continuous batching over the decoder's stream slots.

    requests: list of (prompt [T][NCB+1] int32, n_frames).  A request holds a slot from its prefill
    until it has produced n_frames frames or stopped (im_end); its slot then takes the next waiting
    request.  The active slots are decoded together (one weight read per step) in calls of at most
    frames_per_call frames, cut so that no request overshoots.  expo_fn(request, first_frame, n)
    returns that request's exponential variates [n][11][30] (float32), so a request sees the same
    variates whatever the batch around it.  forced_fn(request, first_frame, n), when given, returns
    that request's forced draws [n][11] (int32; teacher forcing, as in s2_decode_frames).  Returns,
    per request, its codes [NCB][frames] (int32).
    """
    import collections
    import numpy as np
    import torch
    ncb = decoder.d["n_codebooks"]
    waiting = collections.deque(range(len(requests)))
    active = {}
    results = [None] * len(requests)
    while waiting or active:
        for slot in range(slots):
            if slot not in active and waiting:
                r = waiting.popleft()
                decoder.prefill([requests[r][0]], stream_ids=[slot])
                active[slot] = [r, 0, []]
        ids = sorted(active)
        n = min(frames_per_call, min(requests[active[k][0]][1] - active[k][1] for k in ids))
        expo = torch.from_numpy(np.stack([expo_fn(active[k][0], active[k][1], n) for k in ids])).cuda()
        if forced_fn is not None:
            forced = torch.from_numpy(np.stack([forced_fn(active[k][0], active[k][1], n) for k in ids])).cuda()
            out = decoder.decode(n, sampling, expo, forced=forced, stream_ids=ids)
        else:
            out = decoder.decode(n, sampling, expo, stream_ids=ids)
        n_out = out["n_out"].cpu().numpy()
        codes = out["codes"].cpu().numpy()
        for j, k in enumerate(ids):
            r, done, chunks = active[k]
            no = int(n_out[j])
            chunks.append(codes[j, :ncb * no].reshape(ncb, no))
            done += no
            active[k][1] = done
            if no < n or done >= requests[r][1]:
                results[r] = np.concatenate(chunks, axis=1)
                del active[k]
    return results
