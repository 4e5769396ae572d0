"""CUDA path vs oracle on the tiny Dual-AR model (fp32 weights, fp32 KV): whole frames through
the C ABI, teacher-forced with the oracle's own draws, every logit / hidden vector compared at
max-abs-rel <= 1e-4, every draw whose margin exceeds the measured logit error compared exactly,
emitted codes and their layout compared bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.parity import compare_frames, max_abs_rel

pytestmark = pytest.mark.gpu
TOL = 1e-4


def _run(d, w, n_frames, s, prompt, expo, kv_slots=64):
    import dual_ar_tts_gb300 as pkg
    sess = oracle.Session(d, w, kv_slots)
    ref = oracle.generate(sess, prompt, n_frames, s, expo)
    forced = np.zeros((n_frames, 11), np.int32)
    forced[:len(ref["draws"])] = np.asarray(ref["draws"], np.int32)
    dec = pkg.Decoder(d, pkg.upload_weights(w), max_streams=1, kv_slots=kv_slots)
    dec.prefill([prompt])
    out = dec.decode(n_frames, s, torch.from_numpy(expo).cuda()[None], torch.from_numpy(forced).cuda()[None],
                     taps=True)
    assert dec.sync_status() == pkg.S2_OK, pkg.s2_last_error(dec.ctx)
    return ref, out, dec


@pytest.mark.parametrize("jitter,dtype", [(0.0, "f32"), (0.1, "f32"), (0.1, "bf16")])
def test_tiny_frames_match_oracle(jitter, dtype):
    """dtype bf16: the tiny shapes with bf16 weights and an fp16 KV cache, which run the
    tensor-core projection path (tolerance of the bf16 configurations)."""
    cfg = synth.CONFIGS["tiny"]
    d = cfg["dims"] if dtype == "f32" else dict(cfg["dims"], weight_dtype=synth.BF16, kv_dtype=synth.F16)
    tol = TOL if dtype == "f32" else 2e-2
    w = synth.make_weights(d, cfg["weight_seed"], norm_jitter=jitter)
    s = synth.sampling("tiny")
    expo = synth.expo(cfg["input_seed"], 0, cfg["frames"])
    ref, out, dec = _run(d, w, cfg["frames"], s, synth.prompt("tiny"), expo)
    st = compare_frames(ref, out, d, s, tol)
    print(dtype, st)
    assert st["frames"] == cfg["frames"]
    assert st["pinned"] >= 0.9 * st["draws"], st
    dec.close()


def test_tiny_early_stop_and_resume():
    """A main draw of im_end stops the stream (teacher-forced at frame 3): n_out == 3, the codes
    are compacted to the 3 frames produced, and a later call on the stream produces nothing."""
    import dual_ar_tts_gb300 as pkg
    cfg = synth.CONFIGS["tiny"]
    d = cfg["dims"]
    w = synth.make_weights(d, cfg["weight_seed"], norm_jitter=0.1)
    s = synth.sampling("tiny", min_tokens_before_end=0)
    n = 8
    expo = synth.expo(5, 0, n)
    prompt = synth.prompt("tiny")
    free = oracle.generate(oracle.Session(d, w, 64), prompt, n, s, expo)
    forced = np.zeros((n, 11), np.int32)
    forced[:len(free["draws"])] = np.asarray(free["draws"], np.int32)
    forced[3, 0] = d["im_end"]
    ref = oracle.generate(oracle.Session(d, w, 64), prompt, n, s, expo, forced=forced)
    assert ref["stopped"] and len(ref["codes"]) == 3
    dec = pkg.Decoder(d, pkg.upload_weights(w), max_streams=1, kv_slots=64)
    dec.prefill([prompt])
    out = dec.decode(n, s, torch.from_numpy(expo).cuda()[None], torch.from_numpy(forced).cuda()[None], taps=True)
    assert dec.sync_status() == pkg.S2_OK
    compare_frames(ref, out, d, s, TOL)
    assert int(out["n_out"][0]) == 3
    out2 = dec.decode(2, s, torch.from_numpy(synth.expo(6, 0, 2)).cuda()[None], taps=False)
    assert dec.sync_status() == 0
    assert int(out2["n_out"][0]) == 0
    dec.close()


def test_tiny_fast_logits_alone():
    cfg = synth.CONFIGS["tiny"]
    d = cfg["dims"]
    import dual_ar_tts_gb300 as pkg
    w = synth.make_weights(d, 0, norm_jitter=0.1)
    n = 5
    hid, pre = synth.fast_inputs(1, n, d)
    sess = oracle.Session(d, w, 1)
    dec = pkg.Decoder(d, pkg.upload_weights(w), max_streams=1, kv_slots=8)
    got = dec.fast_logits(torch.from_numpy(hid).cuda(), torch.from_numpy(pre).cuda()).cpu().numpy()
    assert dec.sync_status() == 0
    for f in range(n):
        for c in range(1, d["n_codebooks"]):
            ref = sess.fast_logits(hid[f], pre[f, :c])
            assert max_abs_rel(got[f, c - 1], ref) <= TOL
    dec.close()
