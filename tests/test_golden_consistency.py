"""The stored oracle outputs under tests/golden/ (written by make_prefill_golden.py) checked on the
CPU without running the model: they belong to the prompts the generators make today, and the
draws, emitted codes and flat layout follow from the stored logits by the oracle's own draw and
frame bookkeeping (ch.06 §5.1-§5.3 main draw, im_end masking, §6 redraw window, §8 code layout).
A golden file left behind by a change of the generators or of the sampler fails here, before a
GPU test compares against it."""
import numpy as np
import pytest

import oracle
import synth
from tests.golden import make_prefill_golden as golden

CASES = sorted(golden.CASES)


@pytest.fixture(scope="module", params=CASES)
def case(request):
    name = request.param
    c = golden.CASES[name]
    d = golden.case_dims(c)
    prompt, s, expo = golden.case_inputs(c)
    return name, c, d, prompt, s, expo, golden.load(name)


def test_golden_belongs_to_the_current_prompt_and_shape(case):
    name, c, d, prompt, s, expo, ref = case
    assert int(ref["prompt_len"]) == len(prompt)
    assert int(ref["n_layer"]) == d["n_layer"]
    assert int(ref["stream"]) == c["stream"]
    n = golden.N_FRAMES
    adm = oracle.admissible_ids(d)
    assert np.asarray(ref["main_logits"]).shape == (n, adm.size)
    assert np.asarray(ref["hidden"]).shape == (n, d["dim"])
    assert np.asarray(ref["fast_logits"]).shape == (n, d["n_codebooks"] - 1, d["codebook_size"])
    # the first frame draws from the prefill's own outputs
    assert np.array_equal(ref["main_logits"][0], ref["prefill_logits"])
    assert np.array_equal(ref["hidden"][0], ref["prefill_hidden"])
    assert np.isfinite(np.asarray(ref["main_logits"])).all()


def test_golden_draws_and_codes_follow_from_the_stored_logits(case):
    name, c, d, prompt, s, expo, ref = case
    adm = oracle.admissible_ids(d)
    window = []
    codes_all = []
    for f in range(golden.N_FRAMES):
        lg = np.asarray(ref["main_logits"][f], np.float32).copy()
        if f < s["min_tokens_before_end"]:
            lg[-1] = -np.inf  # im_end is the last admissible id
        d0, g0 = oracle.draw(lg, s["temperature"], s["top_p"], s["top_k"], expo[f][0], ids=adm)
        d1, _ = oracle.draw(lg, s["ras_temperature"], s["ras_top_p"], s["top_k"], expo[f][1], ids=adm)
        assert d0 == ref["draws"][f][0], (name, f)
        assert d1 == ref["draws"][f][1], (name, f)
        assert np.allclose(g0, ref["diags"][f][0], rtol=0, atol=0)
        token = d1 if oracle.ras_triggered(d0, window, d) else d0
        codes = [oracle.sem_code(token, d)]
        for cb in range(1, d["n_codebooks"]):
            dc, _ = oracle.draw(ref["fast_logits"][f][cb - 1], s["temperature"], s["top_p"], s["top_k"],
                                expo[f][1 + cb])
            assert dc == ref["draws"][f][1 + cb], (name, f, cb)
            codes.append(dc)
        assert codes == list(ref["codes"][f]), (name, f)
        codes_all.append(codes)
        window = (window + [token])[-s["ras_window"]:]
    assert np.array_equal(oracle.compact(codes_all, d), ref["flat"])
    assert all(0 <= v < d["codebook_size"] for row in codes_all for v in row)
