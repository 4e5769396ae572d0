"""Comparison helpers for CUDA-path vs oracle parity (test support, no arithmetic of the method).

Every ``compare_frames`` call records its statistics in ``REPORT`` (with the test that made it);
``tests/conftest.py`` prints them at the end of the run, so the measured errors of each
configuration stay visible while they are within tolerance, and a drift shows before it fails.
"""
import os

import numpy as np

REPORT = []  # one dict per compare_frames call: test, stream and the statistics it returned


def max_abs_rel(g, r):
    """max_i |g_i - r_i| / max_i |r_i| over finite reference entries."""
    g = np.asarray(g, np.float64)
    r = np.asarray(r, np.float64)
    m = np.isfinite(r)
    den = np.abs(r[m]).max()
    return float(np.abs(g[m] - r[m]).max() / (den if den > 0 else 1.0))


def draw_is_pinned(diag, eps_logit, temperature):
    """A draw must agree when a logit perturbation of at most eps_logit cannot change any of its
    decisions: the top-k cut, the top-p cut and the winner (diag from oracle.draw)."""
    eta = eps_logit / temperature            # perturbation of z = logit / T
    topk_gap, p_gap, best, second = float(diag[0]), float(diag[1]), float(diag[2]), float(diag[3])
    # the variates are indexed by rank, so the winning rank must hold the same token on both
    # sides: its z is apart from the neighbouring ranks' by more than two perturbations
    rank_gap = float(diag[6])
    return topk_gap > 2 * eta and p_gap > 3 * eta and (best - second) > 4 * eta and rank_gap > 2 * eta


def compare_frames(ref, out, d, s, tol, stream=0, check_draws=True):
    """Compare one stream's GPU taps with the oracle trace; returns a dict of statistics and
    raises AssertionError on a violation."""
    n_out = int(out["n_out"][stream])
    assert n_out == len(ref["codes"]), f"frames produced {n_out} vs oracle {len(ref['codes'])}"
    ncb = d["n_codebooks"]
    codes = out["codes"][stream, :ncb * n_out].cpu().numpy()
    assert np.array_equal(codes, ref["flat"]), "emitted codes differ from the oracle"
    ml = out["main_logits"][stream].cpu().numpy()
    hid = out["hidden"][stream].cpu().numpy()
    fl = out["fast_logits"][stream].cpu().numpy()
    dr = out["draws"][stream].cpu().numpy()
    stats = dict(frames=n_out, logit_err=0.0, hidden_err=0.0, fast_err=0.0, draws=0, pinned=0, unpinned=0)
    n_check = len(ref["main_logits"])
    for f in range(n_check):
        e1 = max_abs_rel(ml[f], ref["main_logits"][f])
        e2 = max_abs_rel(hid[f], ref["hidden"][f])
        stats["logit_err"] = max(stats["logit_err"], e1)
        stats["hidden_err"] = max(stats["hidden_err"], e2)
        assert e1 <= tol, f"frame {f}: main logits max-abs-rel {e1:.3g} > {tol}"
        assert e2 <= tol, f"frame {f}: hidden max-abs-rel {e2:.3g} > {tol}"
        eps_main = float(np.abs(ml[f] - ref["main_logits"][f]).max())
        draws_f = ref["draws"][f]
        diags_f = ref["diags"][f]
        for k, gd in enumerate(draws_f):
            if gd < 0:
                continue
            if k >= 2:
                c = k - 1
                fe = fl[f, c - 1]
                rf = ref["fast_logits"][f][c - 1]
                e3 = max_abs_rel(fe, rf)
                stats["fast_err"] = max(stats["fast_err"], e3)
                assert e3 <= tol, f"frame {f} codebook {c}: fast logits max-abs-rel {e3:.3g} > {tol}"
                eps = float(np.abs(fe - rf).max())
                temp = s["temperature"]
            else:
                eps = eps_main
                temp = s["temperature"] if k == 0 else s["ras_temperature"]
            stats["draws"] += 1
            if check_draws and draw_is_pinned(diags_f[k], max(eps, 1e-7), temp):
                stats["pinned"] += 1
                assert int(dr[f, k]) == int(gd), f"frame {f} draw {k}: GPU {dr[f, k]} vs oracle {gd} (pinned)"
            else:
                stats["unpinned"] += 1
    REPORT.append(dict(test=os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0], stream=stream, tol=tol, **stats))
    return stats
