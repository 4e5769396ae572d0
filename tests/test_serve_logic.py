"""Continuous-batching scheduler (dual_ar_tts_gb300.serve) on CPU with a scripted stand-in for the
decoder: slot refilling, calls cut so that no request overshoots, early stops, and per-request
variates indexed by the request's own frame counter."""
import numpy as np
import torch

import dual_ar_tts_gb300 as pkg


class FakeDecoder:
    """Emits code (request * 100 + frame) in every codebook; request 2 stops after 4 frames."""

    def __init__(self, ncb=3):
        self.d = {"n_codebooks": ncb}
        self.slot_req = {}
        self.frames = {}
        self.calls = []

    def prefill(self, prompts, stream_ids):
        (p,), (sid,) = prompts, stream_ids
        self.slot_req[sid] = int(p[0, 0])
        self.frames[sid] = 0

    def decode(self, n, sampling, expo, stream_ids):
        who = [(self.slot_req[sid], self.frames[sid]) for sid in stream_ids]
        self.calls.append((list(stream_ids), n, expo[:, 0, 0, 0].tolist(), who))
        ncb = self.d["n_codebooks"]
        codes = torch.zeros((len(stream_ids), ncb * n), dtype=torch.int32)
        n_out = torch.zeros(len(stream_ids), dtype=torch.int32)
        for j, sid in enumerate(stream_ids):
            r, f0 = self.slot_req[sid], self.frames[sid]
            k = n if r != 2 else max(0, min(n, 4 - f0))
            for cb in range(ncb):
                for f in range(k):
                    codes[j, cb * k + f] = r * 100 + f0 + f
            n_out[j] = k
            self.frames[sid] += k
        return {"codes": codes, "n_out": n_out}


def test_serve_refills_slots_and_cuts_calls():
    reqs = [(np.full((4, 4), r, np.int32), n) for r, n in enumerate([5, 3, 9, 2])]
    expo_fn = lambda r, f0, n: np.full((n, 11, 30), r * 1000 + f0, np.float32)
    orig = torch.Tensor.cuda
    torch.Tensor.cuda = lambda self, *a, **k: self   # the stand-in runs on the host
    try:
        dec = FakeDecoder()
        out = pkg.serve(dec, reqs, slots=2, frames_per_call=3, sampling={}, expo_fn=expo_fn)
    finally:
        torch.Tensor.cuda = orig
    lens = [o.shape[1] for o in out]
    assert lens == [5, 3, 4, 2]                  # request 2 stopped after 4 frames
    for r, o in enumerate(out):
        assert o.shape[0] == 3
        np.testing.assert_array_equal(o[0], r * 100 + np.arange(lens[r]))
    for ids, n, first, who in dec.calls:
        assert 1 <= n <= 3
        for v, (r, f0) in zip(first, who):
            assert int(v) == r * 1000 + f0           # the request's own variates, at its own frame
    # the first call holds requests 0 and 1 and is cut to request 1's 3 frames
    assert dec.calls[0][0] == [0, 1] and dec.calls[0][1] == 3
