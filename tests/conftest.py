import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running (full-size workloads)")


def pytest_terminal_summary(terminalreporter):
    """The parity statistics of the run (tests.parity.REPORT): per compared stream, the largest
    max-abs-rel of the main logits, hidden state and Fast-AR logits against the oracle, the
    tolerance, and the draws compared (pinned ones must be equal, the rest are teacher-forced).
    With S2_PARITY_REPORT set, also written there as JSON."""
    from tests import parity
    if not parity.REPORT:
        return
    tr = terminalreporter
    tr.write_sep("-", "parity with the oracle (max-abs-rel; draws pinned / compared)")
    try:
        for r in parity.REPORT:
            tr.write_line(f"{r['test']} [stream {r['stream']}]: logits {r['logit_err']:.2e}  "
                          f"hidden {r['hidden_err']:.2e}  fast {r['fast_err']:.2e}  (tol {r['tol']:.0e}); "
                          f"frames {r['frames']}, draws {r['pinned']} / {r['draws']}")
        path = os.environ.get("S2_PARITY_REPORT")
        if path:
            import json
            with open(path, "w") as f:
                json.dump(parity.REPORT, f, indent=1)
    except Exception as e:  # a report problem must not change the run's outcome
        tr.write_line(f"(parity report incomplete: {e!r})")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


@pytest.fixture(scope="session")
def s2pro():
    """S2-Pro-shaped synthetic weights (seed 0): dims, host arrays, device tensors, names."""
    import torch
    import synth
    import dual_ar_tts_gb300 as pkg
    d = synth.CONFIGS["frame"]["dims"]
    host = synth.make_weights(d, 0)
    dev = pkg.upload_weights(host)
    names = [n for n, _, _ in synth.weight_specs(d)]
    yield d, host, dev, names
    del dev
    torch.cuda.empty_cache()
