"""The batch-1 kernel's grid barrier across the 2^32 wrap of its counter.

The counter grows by the grid size at every phase, so a long Fast-AR-alone call wraps it.  A
testing hook starts the counter a few phases below 2^32; the results must still equal the
oracle's (Fast-AR alone and whole frames), which they cannot if a CTA passes a barrier early, and
the Fast-AR logits must be bit-identical to a call that starts the counter at 0.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.parity import compare_frames, max_abs_rel

pytestmark = pytest.mark.gpu
NEAR_WRAP = 2 ** 32 - 1000


def test_tiny_fast_alone_across_counter_wrap():
    import dual_ar_tts_gb300 as pkg
    d = synth.CONFIGS["tiny"]["dims"]
    w = synth.make_weights(d, 0, norm_jitter=0.1)
    n = 4
    hid, pre = synth.fast_inputs(2, n, d)
    sess = oracle.Session(d, w, 1)
    dec = pkg.Decoder(d, pkg.upload_weights(w), max_streams=1, kv_slots=8)
    pkg.s2_set_barrier_base(dec.ctx, NEAR_WRAP)
    got = dec.fast_logits(torch.from_numpy(hid).cuda(), torch.from_numpy(pre).cuda()).cpu().numpy()
    assert dec.sync_status() == pkg.S2_OK, pkg.s2_last_error(dec.ctx)
    for f in range(n):
        for c in range(1, d["n_codebooks"]):
            assert max_abs_rel(got[f, c - 1], sess.fast_logits(hid[f], pre[f, :c])) <= 1e-4, (f, c)
    dec.close()


def test_tiny_frames_across_counter_wrap():
    import dual_ar_tts_gb300 as pkg
    cfg = synth.CONFIGS["tiny"]
    d = cfg["dims"]
    w = synth.make_weights(d, 0, norm_jitter=0.1)
    n = 4
    s = synth.sampling("tiny", min_tokens_before_end=n)
    expo = synth.expo(8, 0, n)
    prompt = synth.prompt("tiny")
    ref = oracle.generate(oracle.Session(d, w, 64), prompt, n, s, expo)
    forced = np.asarray(ref["draws"], np.int32)
    dec = pkg.Decoder(d, pkg.upload_weights(w), max_streams=1, kv_slots=64)
    dec.prefill([prompt])
    pkg.s2_set_barrier_base(dec.ctx, NEAR_WRAP)
    out = dec.decode(n, s, torch.from_numpy(expo).cuda()[None], torch.from_numpy(forced).cuda()[None], taps=True)
    assert dec.sync_status() == pkg.S2_OK, pkg.s2_last_error(dec.ctx)
    compare_frames(ref, out, d, s, 1e-4)
    dec.close()


def test_s2pro_fast_alone_across_counter_wrap(s2pro):
    import dual_ar_tts_gb300 as pkg
    _, host, dev, names = s2pro
    d = synth.CONFIGS["fast"]["dims"]
    by_h, by_d = dict(zip(names, host)), dict(zip(names, dev))
    wh = [None if n in ("embeddings", "codebook_embeddings", "norm") else by_h[n] for n, _, _ in synth.weight_specs(d)]
    wd = [None if n in ("embeddings", "codebook_embeddings", "norm") else by_d[n] for n, _, _ in synth.weight_specs(d)]
    n = 3
    hid, pre = synth.fast_inputs(7, n, d)
    dec = pkg.Decoder(d, wd, max_streams=1, kv_slots=0)
    h, p = torch.from_numpy(hid).cuda(), torch.from_numpy(pre).cuda()
    base = dec.fast_logits(h, p).clone()
    pkg.s2_set_barrier_base(dec.ctx, NEAR_WRAP)
    wrapped = dec.fast_logits(h, p).clone()
    assert dec.sync_status() == pkg.S2_OK, pkg.s2_last_error(dec.ctx)
    assert torch.equal(base, wrapped)
    sess = oracle.Session(d, wh, 1)
    got = wrapped.cpu().numpy()
    for c in (1, 5, 9):
        assert max_abs_rel(got[n - 1, c - 1], sess.fast_logits(hid[n - 1], pre[n - 1, :c])) <= 2e-2
    dec.close()
