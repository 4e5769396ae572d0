"""s2_fast_logits_static — Fast-AR alone on the library's static scratch (no allocation).

It serves callers that cannot allocate device memory: an application whose memory pool already
holds the device, or a latency-critical thread that must not block in cudaMalloc/cudaFree.

The GPU test calls the static entry point through the C ABI twice in a row, with different inputs
and frame counts, and compares each output with s2_fast_logits of a context on the same weights
and with the oracle (same tolerances as the other parity tests: 1e-4 for fp32 weights, 2e-2 for
bf16).  A second test checks that a repeated call changes neither the device's free memory nor
the memory torch has allocated.  The file is named to be collected last, and passes alone in a
fresh process as well as after the other tests.  The CPU tests check the argument and size
rejections, which return before any CUDA call.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
from tests.parity import max_abs_rel


@pytest.fixture(scope="module")
def pkg():
    from dual_ar_tts_gb300 import build
    build.build()
    import dual_ar_tts_gb300 as p
    p.load()
    return p


def _ptrs(tensors):
    return [t.data_ptr() if t is not None else 0 for t in tensors]


@pytest.mark.gpu
@pytest.mark.parametrize("case,tol", [("tiny", 1e-4), ("fast", 2e-2)])
def test_static_matches_context_path_on_two_calls(pkg, case, tol):
    d = synth.CONFIGS[case]["dims"]
    host = synth.make_weights(d, 0, norm_jitter=0.1 if case == "tiny" else 0.0)
    dev = pkg.upload_weights(host)
    dims = pkg.make_dims(d)
    dec = pkg.Decoder(d, dev, max_streams=1, kv_slots=8 if d["n_layer"] > 0 else 0)
    sess = oracle.Session(d, host, 1)
    stream = torch.cuda.current_stream().cuda_stream
    ncb, cbs = d["n_codebooks"], d["codebook_size"]
    for seed, n in ((11, 8), (12, 5)):
        hid, pre = synth.fast_inputs(seed, n, d)
        h = torch.from_numpy(hid).cuda()
        p = torch.from_numpy(pre).cuda()
        out = torch.full((n, ncb - 1, cbs), float("nan"), device="cuda")
        status = torch.full((2,), -1, dtype=torch.int32, device="cuda")
        pkg.s2_fast_logits_static(dims, _ptrs(dev), n, h.data_ptr(), p.data_ptr(), out.data_ptr(),
                                  status.data_ptr(), stream)
        ref = dec.fast_logits(h, p)
        assert dec.sync_status() == pkg.S2_OK, pkg.s2_last_error(dec.ctx)
        assert int(status[0].item()) == pkg.S2_OK, status.tolist()
        got, want = out.cpu().numpy(), ref.cpu().numpy()
        assert np.isfinite(got).all()
        worst = max(max_abs_rel(got[f, c], want[f, c]) for f in range(n) for c in range(ncb - 1))
        assert worst <= tol, (case, seed, worst)
        # the oracle recomputes each window from scratch (first and last frame, three windows)
        for f in (0, n - 1):
            for c in (1, (ncb - 1) // 2 + 1, ncb - 1):
                e = max_abs_rel(got[f, c - 1], sess.fast_logits(hid[f], pre[f, :c]))
                assert e <= tol, (case, seed, f, c, e)
    dec.close()


@pytest.mark.gpu
def test_static_repeat_call_allocates_no_device_memory(pkg):
    d = synth.CONFIGS["tiny"]["dims"]
    dev = pkg.upload_weights(synth.make_weights(d, 0, norm_jitter=0.1))
    dims = pkg.make_dims(d)
    stream = torch.cuda.current_stream().cuda_stream
    ncb, cbs = d["n_codebooks"], d["codebook_size"]
    n = 6
    hid, pre = synth.fast_inputs(21, n, d)
    h = torch.from_numpy(hid).cuda()
    p = torch.from_numpy(pre).cuda()
    out = torch.empty((n, ncb - 1, cbs), device="cuda")
    status = torch.empty((2,), dtype=torch.int32, device="cuda")
    # the first call with this weight table sets the array up
    pkg.s2_fast_logits_static(dims, _ptrs(dev), n, h.data_ptr(), p.data_ptr(), out.data_ptr(), status.data_ptr(),
                              stream)
    torch.cuda.synchronize()
    first = out.clone()
    free0, _ = torch.cuda.mem_get_info()
    alloc0 = torch.cuda.memory_allocated()
    out.fill_(float("nan"))
    torch.cuda.synchronize()
    pkg.s2_fast_logits_static(dims, _ptrs(dev), n, h.data_ptr(), p.data_ptr(), out.data_ptr(), status.data_ptr(),
                              stream)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, (free0, free1)
    assert torch.cuda.memory_allocated() == alloc0
    assert int(status[0].item()) == pkg.S2_OK
    assert torch.equal(out, first)


def test_static_rejects_bad_arguments_before_any_cuda_call(pkg):
    d = synth.CONFIGS["tiny"]["dims"]
    dims = pkg.make_dims(d)
    n_w = len(synth.weight_specs(d))
    fake = [16 * (i + 1) for i in range(n_w)]  # never dereferenced: every case fails its checks first
    lib = pkg.load()
    arr = (ctypes.c_void_p * n_w)(*fake)
    assert lib.s2_fast_logits_static(ctypes.byref(dims), arr, n_w - 1, 1, 16, 16, 16, None, None) == pkg.S2_EINVAL
    assert lib.s2_fast_logits_static(ctypes.byref(dims), arr, n_w, 0, 16, 16, 16, None, None) == pkg.S2_EINVAL
    assert lib.s2_fast_logits_static(ctypes.byref(dims), arr, n_w, 1, None, 16, 16, None, None) == pkg.S2_EINVAL
    bad = list(fake)
    bad[-1] = 24  # not 16-byte aligned
    arr_bad = (ctypes.c_void_p * n_w)(*bad)
    assert lib.s2_fast_logits_static(ctypes.byref(dims), arr_bad, n_w, 1, 16, 16, 16, None, None) == pkg.S2_EINVAL
    assert "aligned" in pkg.s2_last_error(None)


@pytest.mark.parametrize("over,limit", [
    # a Fast-AR decoder with more phases than the static program holds (16 layers, 15 codebooks)
    (dict(fast_dim=5120, dim=5120, fast_ffn=5120, fast_n_layer=16, fast_n_head=40, fast_n_kv_head=10,
          n_codebooks=15, fast_window=16), "1024"),
    # one whose scratch exceeds the array (12 wide layers: within-frame K/V and SwiGLU buffers)
    (dict(fast_dim=5120, dim=5120, fast_ffn=20480, fast_n_layer=12, fast_n_head=40, fast_n_kv_head=10),
     str(2 << 20)),
])
def test_static_rejects_shapes_beyond_its_limits(pkg, over, limit):
    d = dict(synth.CONFIGS["fast"]["dims"])
    d.update(over)
    dims = pkg.make_dims(d)
    lib = pkg.load()
    n_w = lib.s2_weight_count(ctypes.byref(dims))
    assert n_w > 0
    arr = (ctypes.c_void_p * n_w)(*[16 * (i + 1) for i in range(n_w)])
    rc = lib.s2_fast_logits_static(ctypes.byref(dims), arr, n_w, 1, 16, 16, 16, None, None)
    assert rc == pkg.S2_ENOMEM
    msg = pkg.s2_last_error(None)
    assert "static" in msg and limit in msg, msg
