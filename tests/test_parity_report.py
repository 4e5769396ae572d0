"""The comparison helper itself (tests.parity.compare_frames), on hand-made traces: what it
accepts, what it rejects, and the statistics it records for the end-of-run parity summary."""
import numpy as np
import pytest
import torch

from tests import parity

D = dict(n_codebooks=3)
S = dict(temperature=0.7, ras_temperature=1.0)


def _trace(n_frames=2, seed=0):
    rng = np.random.default_rng(seed)
    ml = [rng.standard_normal(16).astype(np.float32) for _ in range(n_frames)]
    hid = [rng.standard_normal(8).astype(np.float32) for _ in range(n_frames)]
    fl = [np.stack([rng.standard_normal(5).astype(np.float32) for _ in range(2)]) for _ in range(n_frames)]
    draws = [[1, -1, 2, 3] for _ in range(n_frames)]
    # diagnostics: top-k gap, top-p gap, best, second, -, -, rank gap (all large: every draw pinned)
    diags = [[[1.0, 1.0, 5.0, 1.0, 0.0, 0.0, 1.0]] * 4 for _ in range(n_frames)]
    codes = [[4, 5, 6] for _ in range(n_frames)]
    ref = dict(main_logits=ml, hidden=hid, fast_logits=fl, draws=draws, diags=diags, codes=codes,
               flat=np.asarray(codes, np.int32).T.reshape(-1))
    out = dict(n_out=torch.tensor([n_frames]),
               codes=torch.from_numpy(ref["flat"].copy())[None],
               main_logits=torch.from_numpy(np.stack(ml))[None],
               hidden=torch.from_numpy(np.stack(hid))[None],
               fast_logits=torch.from_numpy(np.stack(fl))[None],
               draws=torch.from_numpy(np.asarray([[1, -1, 2, 3]] * n_frames, np.int32))[None])
    return ref, out


def test_identical_trace_passes_and_is_recorded():
    ref, out = _trace()
    n0 = len(parity.REPORT)
    st = parity.compare_frames(ref, out, D, S, 1e-4)
    assert st["logit_err"] == 0.0 and st["hidden_err"] == 0.0 and st["fast_err"] == 0.0
    assert st["draws"] == 6 and st["pinned"] == 6
    assert len(parity.REPORT) == n0 + 1
    rec = parity.REPORT[-1]
    assert rec["test"].endswith("test_identical_trace_passes_and_is_recorded") and rec["tol"] == 1e-4
    parity.REPORT.pop()


@pytest.mark.parametrize("what", ["main_logits", "hidden", "fast_logits", "draws", "codes"])
def test_each_kind_of_difference_is_rejected(what):
    ref, out = _trace()
    n0 = len(parity.REPORT)
    if what == "draws":
        out["draws"][0, 1, 2] = 4            # a pinned Fast-AR draw differs
    elif what == "codes":
        out["codes"][0, 3] += 1
    elif what == "fast_logits":
        out["fast_logits"][0, 0, 1, 2] += 1.0
    else:
        out[what][0, 1, 3] += 1.0
    with pytest.raises(AssertionError):
        parity.compare_frames(ref, out, D, S, 1e-4)
    assert len(parity.REPORT) == n0  # a failed comparison records nothing


def test_small_error_within_tolerance_is_measured():
    ref, out = _trace()
    out["hidden"][0, 0] *= 1.0 + 1e-6
    st = parity.compare_frames(ref, out, D, S, 1e-4)
    assert 0.0 < st["hidden_err"] <= 1e-5
    parity.REPORT.pop()
