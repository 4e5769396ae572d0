"""Failure detection without a GPU fault: every device-side wait is bounded.  A tiny wait bound
makes some wait give up; the call must report S2_ETIMEOUT through s2_sync_status (no trap, no
fault), and the context must decode normally once the default bound is restored."""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


def test_wait_bound_gives_timeout_status_and_the_context_recovers():
    import dual_ar_tts_gb300 as pkg
    cfg = synth.CONFIGS["tiny"]
    d = cfg["dims"]
    dec = pkg.Decoder(d, pkg.upload_weights(synth.make_weights(d, cfg["weight_seed"])), max_streams=1, kv_slots=64)
    prompt = synth.prompt("tiny")
    s = synth.sampling("tiny", min_tokens_before_end=1000)
    n = 6
    expo = torch.from_numpy(synth.expo(cfg["input_seed"], 0, n)).cuda()[None]

    dec.prefill([prompt])
    pkg.s2_set_spin_limit(dec.ctx, 1)  # about 1 us: a grid barrier or pipeline wait gives up
    dec.decode(n, s, expo)
    assert dec.sync_status() == pkg.S2_ETIMEOUT
    msg = pkg.s2_last_error(dec.ctx)
    assert "gave up" in msg
    # the report names the wait, the CTA and (for the consumers' waits) the phase of the launch
    import re
    m = re.search(r"site (\d+), CTA (\d+)(, phase (\d+) of the launch)?\)", msg)
    assert m, msg
    assert 0 <= int(m.group(2)) < 1024
    if m.group(4) is not None:
        assert 0 <= int(m.group(4)) < n * pkg.s2_phase_count(dec.ctx)

    pkg.s2_set_spin_limit(dec.ctx, 0)  # the default bound again
    dec.prefill([prompt])
    out = dec.decode(n, s, expo)
    assert dec.sync_status() == pkg.S2_OK, pkg.s2_last_error(dec.ctx)
    assert int(out["n_out"][0]) == n
    codes = out["codes"].cpu().numpy().reshape(d["n_codebooks"], n)
    assert (codes >= 0).all() and (codes < d["codebook_size"]).all()
    # the same call from the same state gives the same codes (nothing left over from the failure)
    dec.prefill([prompt])
    again = dec.decode(n, s, expo)
    assert dec.sync_status() == pkg.S2_OK
    assert np.array_equal(again["codes"].cpu().numpy(), out["codes"].cpu().numpy())
