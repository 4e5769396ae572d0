"""CUDA path vs oracle at S2-Pro shapes (bf16 weights, fp16 KV cache), through the C ABI.

* Fast-AR alone: 1000 teacher-forced frames x 9 windows on the GPU; the oracle recomputes each
  window from scratch (no prefix cache) on a sample of frames; logits max-abs-rel <= 2e-2.
* Full frame, batch 1: the 512-position prompt, then 40 frames teacher-forced with the oracle's
  own draws (past min_tokens_before_end = 32, where im_end becomes drawable); Slow-AR logits
  (admissible ids), hidden state and every Fast-AR logit vector compared at max-abs-rel <= 2e-2,
  pinned draws and all emitted codes compared exactly.
* Full frame at its bench length (256 frames, free running): properties that hold at any size —
  every frame produced, codes in range, identical codes on a second run from the same state.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.parity import compare_frames, max_abs_rel

pytestmark = pytest.mark.gpu
TOL = 2e-2


def _subset(names_full, tensors, d_sub):
    by = dict(zip(names_full, tensors))
    return [None if (d_sub["n_layer"] == 0 and n in ("embeddings", "codebook_embeddings", "norm")) else by[n]
            for n, _, _ in synth.weight_specs(d_sub)]


def test_fast_alone_1000_frames(s2pro):
    import dual_ar_tts_gb300 as pkg
    d_full, host, dev, names = s2pro
    cfg = synth.CONFIGS["fast"]
    d = cfg["dims"]
    n = cfg["frames"]
    hid, pre = synth.fast_inputs(cfg["input_seed"], n, d)
    dec = pkg.Decoder(d, _subset(names, dev, d), max_streams=1, kv_slots=0)
    got = dec.fast_logits(torch.from_numpy(hid).cuda(), torch.from_numpy(pre).cuda())
    assert dec.sync_status() == pkg.S2_OK, pkg.s2_last_error(dec.ctx)
    got = got.cpu().numpy()
    assert np.isfinite(got).all()
    sess = oracle.Session(d, _subset(names, host, d), 1)
    worst = 0.0
    for f in list(range(4)) + list(range(100, n, 150)):
        for c in range(1, d["n_codebooks"]):
            ref = sess.fast_logits(hid[f], pre[f, :c])
            e = max_abs_rel(got[f, c - 1], ref)
            worst = max(worst, e)
            assert e <= TOL, (f, c, e)
    print(f"fast-alone worst max-abs-rel {worst:.3g}")
    dec.close()


def test_full_frame_prefill_and_frames_match_oracle(s2pro):
    import dual_ar_tts_gb300 as pkg
    d, host, dev, names = s2pro
    cfg = synth.CONFIGS["frame"]
    n_frames = 40
    prompt = synth.prompt("frame")
    s = synth.sampling("frame")
    expo = synth.expo(cfg["input_seed"], 0, n_frames)
    sess = oracle.Session(d, host, len(prompt) + n_frames + 1)
    ref = oracle.generate(sess, prompt, n_frames, s, expo)
    forced = np.zeros((n_frames, 11), np.int32)
    forced[:len(ref["draws"])] = np.asarray(ref["draws"], np.int32)
    dec = pkg.Decoder(d, dev, max_streams=1, kv_slots=1024)
    dec.prefill([prompt])
    out = dec.decode(n_frames, s, torch.from_numpy(expo).cuda()[None], torch.from_numpy(forced).cuda()[None],
                     taps=True)
    assert dec.sync_status() == pkg.S2_OK, pkg.s2_last_error(dec.ctx)
    st = compare_frames(ref, out, d, s, TOL)
    print("full-frame parity:", st)
    dec.close()


def test_full_frame_bench_length_properties(s2pro):
    import dual_ar_tts_gb300 as pkg
    d, host, dev, names = s2pro
    cfg = synth.CONFIGS["frame"]
    K = cfg["frames"]
    prompt = synth.prompt("frame")
    s = synth.sampling("frame", min_tokens_before_end=K)
    expo = torch.from_numpy(synth.expo(cfg["input_seed"], 0, K)).cuda()[None]
    runs = []
    for _ in range(2):
        dec = pkg.Decoder(d, dev, max_streams=1, kv_slots=1024)
        dec.prefill([prompt])
        out = dec.decode(K, s, expo, taps=True)
        assert dec.sync_status() == pkg.S2_OK, pkg.s2_last_error(dec.ctx)
        runs.append({k: v.cpu() for k, v in out.items()})
        dec.close()
    a, b = runs
    assert int(a["n_out"][0]) == K
    codes = a["codes"][0].numpy().reshape(d["n_codebooks"], K)
    assert (codes >= 0).all() and (codes < d["codebook_size"]).all()
    assert torch.equal(a["codes"], b["codes"]) and torch.equal(a["draws"], b["draws"])
    assert torch.isfinite(a["main_logits"]).all() and torch.isfinite(a["fast_logits"]).all()
    # main draws are admissible ids, fast draws are codes
    dr = a["draws"][0].numpy()
    assert ((dr[:, 0] >= d["sem_begin"]) & (dr[:, 0] <= d["sem_end"])).all()
    assert ((dr[:, 2:11] >= 0) & (dr[:, 2:11] < d["codebook_size"])).all()
