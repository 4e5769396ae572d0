"""The C-ABI library builds, loads without a GPU, exports every entry point the header declares,
and its host-side logic (weight table, workspace sizing, argument checks) agrees with the
generator's weight table."""
import ctypes
import os
import re
import subprocess

import pytest

import numpy as np
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "s2frame.h")


@pytest.fixture(scope="module")
def lib():
    from dual_ar_tts_gb300 import build
    build.build()
    import dual_ar_tts_gb300 as pkg
    return pkg.load()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(s2_[a-z0-9_]+)\s*\(", text)))


def test_header_declarations_are_exported(lib):
    names = _declared()
    assert "s2_decode_frames" in names and "s2_frame_init" in names
    so = os.path.join(ROOT, "dual_ar_tts_gb300", "libs2frame.so")
    syms = subprocess.run(["nm", "-D", "--defined-only", so], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (s2_\w+)", syms))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        assert hasattr(lib, n)
    import dual_ar_tts_gb300 as pkg
    assert set(pkg.EXPORTS) == set(names)


@pytest.mark.parametrize("cfg", ["tiny", "frame", "fast"])
def test_weight_table_matches_generator(lib, cfg):
    import dual_ar_tts_gb300 as pkg
    d = synth.CONFIGS[cfg]["dims"]
    dims = pkg.make_dims(d)
    specs = synth.weight_specs(d)
    assert pkg.s2_weight_count(dims) == len(specs)
    for i, (name, shape, _) in enumerate(specs):
        nm, n = pkg.s2_weight_info(dims, i)
        assert nm == name
        assert n == int(__import__("numpy").prod(shape))
    assert pkg.s2_weight_info(dims, len(specs))[1] == -1


def test_workspace_sizing_and_bad_dims(lib):
    import dual_ar_tts_gb300 as pkg
    d = synth.CONFIGS["frame"]["dims"]
    one = pkg.s2_frame_workspace_bytes(pkg.make_dims(d), 1, 32768)
    kv = 2 * 36 * 8 * 32768 * 128 * 2
    assert kv < one < kv + 2 ** 30
    assert pkg.s2_frame_workspace_bytes(pkg.make_dims(d), 2, 32768) > one + kv // 2
    bad = dict(d, head_dim=96)
    assert pkg.s2_frame_workspace_bytes(pkg.make_dims(bad), 1, 16) == 0
    bad = dict(d, fast_n_layer=0)                  # no fast decoder (ch.06 §1 entry check)
    assert pkg.s2_weight_count(pkg.make_dims(bad)) == -1
    bad = dict(d, fast_window=9)                   # window must hold the 10 codebook positions
    assert pkg.s2_weight_count(pkg.make_dims(bad)) == -1


def test_init_rejects_bad_arguments_without_touching_a_gpu(lib):
    import dual_ar_tts_gb300 as pkg
    d = synth.CONFIGS["tiny"]["dims"]
    dims = pkg.make_dims(d)
    n = pkg.s2_weight_count(dims)
    out = ctypes.c_void_p()
    arr = (ctypes.c_void_p * (n - 1))()
    rc = lib.s2_frame_init(ctypes.byref(dims), arr, n - 1, ctypes.c_void_p(256), 1 << 20, 1, 64, ctypes.byref(out))
    assert rc == pkg.S2_EINVAL and "weight table" in pkg.s2_last_error(None)
    arr = (ctypes.c_void_p * n)(*([256] * n))
    rc = lib.s2_frame_init(ctypes.byref(dims), arr, n, ctypes.c_void_p(8), 1 << 20, 1, 64, ctypes.byref(out))
    assert rc == pkg.S2_EINVAL and "aligned" in pkg.s2_last_error(None)


def test_codec_latent_rejects_bad_arguments_before_any_cuda_call():
    import ctypes
    import dual_ar_tts_gb300 as pkg
    lib = pkg.load()
    arr = (ctypes.c_void_p * 2)(16, 32)
    assert lib.s2_codec_latent(2, 64, 12, arr, 4, 16, 16, None, None) == pkg.S2_EINVAL   # dim not a multiple of 8
    assert lib.s2_codec_latent(0, 64, 16, arr, 4, 16, 16, None, None) == pkg.S2_EINVAL   # no codebook
    assert lib.s2_codec_latent(2, 64, 16, arr, 0, 16, 16, None, None) == pkg.S2_EINVAL   # no frame
    bad = (ctypes.c_void_p * 2)(16, 40)                                                  # unaligned quantizer
    assert lib.s2_codec_latent(2, 64, 16, bad, 4, 16, 16, None, None) == pkg.S2_EINVAL


def test_quantize_e4m3_rejects_bad_arguments_before_any_cuda_call():
    import dual_ar_tts_gb300 as pkg
    lib = pkg.load()
    assert lib.s2_quantize_e4m3(16, 0, 8, 32, 64, None) == pkg.S2_EINVAL    # no row
    assert lib.s2_quantize_e4m3(16, 4, 0, 32, 64, None) == pkg.S2_EINVAL    # no column
    assert lib.s2_quantize_e4m3(None, 4, 8, 32, 64, None) == pkg.S2_EINVAL  # no matrix
    assert lib.s2_quantize_e4m3(17, 4, 8, 32, 64, None) == pkg.S2_EINVAL    # unaligned bf16 rows
    assert lib.s2_quantize_e4m3(16, 4, 8, 32, 66, None) == pkg.S2_EINVAL    # unaligned scales


def test_draw_rejects_bad_arguments_before_any_cuda_call():
    import dual_ar_tts_gb300 as pkg
    lib = pkg.load()
    assert lib.s2_draw(0, 16, 64, -1, 0, 0, 0.7, 0.8, 32, 48, None) == pkg.S2_EINVAL      # no row
    assert lib.s2_draw(1, 16, 0, -1, 0, 0, 0.7, 0.8, 32, 48, None) == pkg.S2_EINVAL       # empty row
    assert lib.s2_draw(1, 16, 4353, -1, 0, 0, 0.7, 0.8, 32, 48, None) == pkg.S2_EINVAL    # row too long
    assert lib.s2_draw(1, 16, 1, 100, 7, 0, 0.7, 0.8, 32, 48, None) == pkg.S2_EINVAL      # main row without im_end
    assert lib.s2_draw(1, None, 64, -1, 0, 0, 0.7, 0.8, 32, 48, None) == pkg.S2_EINVAL    # no logits
    assert lib.s2_draw(1, 16, 64, -1, 0, 0, 0.7, 0.8, None, 48, None) == pkg.S2_EINVAL    # no variates
    assert lib.s2_draw(1, 16, 64, -1, 0, 0, 0.7, 0.8, 32, None, None) == pkg.S2_EINVAL    # no output
    assert lib.s2_draw(1, 18, 64, -1, 0, 0, 0.7, 0.8, 32, 48, None) == pkg.S2_EINVAL      # unaligned logits
    assert lib.s2_draw(1, 16, 64, -1, 0, 0, 0.0, 0.8, 32, 48, None) == pkg.S2_EINVAL      # temperature 0
    assert lib.s2_draw(1, 16, 64, -1, 0, 0, -1.0, 0.8, 32, 48, None) == pkg.S2_EINVAL     # negative temperature
    assert lib.s2_draw(1, 16, 64, -1, 0, 0, float("nan"), 0.8, 32, 48, None) == pkg.S2_EINVAL
    assert lib.s2_draw(1, 16, 64, -1, 0, 0, 0.7, float("inf"), 32, 48, None) == pkg.S2_EINVAL


def test_fp8_dims_are_checked():
    import dual_ar_tts_gb300 as pkg
    import synth
    d = dict(synth.CONFIGS["tiny"]["dims"], weight_fp8=1)        # fp32 weights
    assert pkg.s2_frame_workspace_bytes(pkg.make_dims(d), 1, 64) == 0
    d = dict(synth.MINI, weight_fp8=1, ffn=576)                 # 576 is not a multiple of 128
    assert pkg.s2_frame_workspace_bytes(pkg.make_dims(d), 1, 64) == 0
    d = dict(synth.MINI, weight_fp8=2)
    assert pkg.s2_frame_workspace_bytes(pkg.make_dims(d), 1, 64) == 0
    d8 = dict(synth.MINI, weight_fp8=1)
    a = pkg.s2_frame_workspace_bytes(pkg.make_dims(synth.MINI), 2, 64)
    b = pkg.s2_frame_workspace_bytes(pkg.make_dims(d8), 2, 64)
    # the e4m3 copies of the projections (1 byte per element + a 4-byte scale per row) are carved too
    import oracle
    host_shapes = [s for _, s, _ in synth.weight_specs(synth.MINI)]
    q = sum(int(np.prod(host_shapes[i])) + 4 * host_shapes[i][0] for i in oracle.projection_indices(synth.MINI))
    assert q <= b - a <= q + 256 * (2 * len(oracle.projection_indices(synth.MINI)) + 1)


def test_static_fast_logits_rejects_fp8_dims_before_any_cuda_call():
    import dual_ar_tts_gb300 as pkg
    import synth
    d = dict(synth.MINI, weight_fp8=1)
    n = pkg.s2_weight_count(pkg.make_dims(d))
    with pytest.raises(pkg.S2Error) as e:
        pkg.s2_fast_logits_static(pkg.make_dims(d), [16] * n, 1, 16, 16, 16)
    assert e.value.code == pkg.S2_EINVAL
