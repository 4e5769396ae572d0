"""The device draw (s2_draw, the routine both decode engines run) against the oracle's draw on
crafted logits rows.

The draw (s2.cpp analysis ch.06 "Fast-AR codebook decoding and the generation main loop" §5; the
Mizuoto "Fish Speech" engine page): top 30 of z = logit / T by (z desc, id asc), softmax over them,
rank r kept iff r == 0 or Σ_{s<r} π_s < top_p, winner = argmax π_r / E_r.  Both sides take z with
the same fp32 division, so the candidate set and its order are exact; only π goes through expf,
whose last-place rounding may differ between CUDA and the host C library.  A row is therefore
compared where the oracle's top-p cut and its winning score stand more than 1e-5 from a tie (with
all-equal logits π is exact and every such row is compared).

Rows: Gaussian; quantised to steps of 1/2 and 1 (ties at the top-30 cut, and more than 64 keys at
or above the selection threshold, which takes the histogram selection); all equal (+0: the
histogram selection with 4096 equal keys at S2-Pro width, the threshold selection at 64); signed
zeros (-0 and +0 tie); sparse valid entries (-inf elsewhere), fewer than 30 valid, none valid
(-1); NaN and +inf entries (not drawable); huge and subnormal magnitudes; main rows with im_end
as the largest logit, masked (min_tokens) or not.  Lengths: S2-Pro's 4096 codes and 4097
admissible main entries, the tiny model's 64 and 65, the 4352 maximum and a single entry.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

S2PRO_MAIN = dict(sem_begin=151678, im_end=151645)   # im_end below the semantic range
TINY_MAIN = dict(sem_begin=4096, im_end=4160)        # im_end above it
ROWS = 24


def _rows(kind, n, rng):
    x = rng.standard_normal((ROWS, n)).astype(np.float32) * 3.0
    if kind == "gauss":
        return x
    if kind == "half":
        return (np.round(x * 2) / 2).astype(np.float32)
    if kind == "unit":
        return np.round(x).astype(np.float32)
    if kind == "equal":
        return np.zeros((ROWS, n), np.float32)
    if kind == "signed_zero":
        z = np.zeros((ROWS, n), np.float32)
        z[:, 1::2] = -0.0
        return z
    if kind == "sparse":
        keep = rng.random((ROWS, n)) < 0.01
        keep[:, 0] = True
        return np.where(keep, x, -np.inf).astype(np.float32)
    if kind == "few":
        out = np.full((ROWS, n), -np.inf, np.float32)
        for r in range(ROWS):
            idx = rng.choice(n, size=min(n, 1 + r % 7), replace=False)
            out[r, idx] = x[r, idx]
        return out
    if kind == "none":
        return np.full((ROWS, n), -np.inf, np.float32)
    if kind == "nonfinite":
        y = x.copy()
        y[rng.random((ROWS, n)) < 0.1] = np.nan
        y[rng.random((ROWS, n)) < 0.02] = np.inf
        return y
    if kind == "magnitude":
        y = x.copy()
        y[:, ::3] *= np.float32(1e30)
        y[:, 1::3] *= np.float32(1e-42)
        return y
    raise ValueError(kind)


KINDS = ["gauss", "half", "unit", "equal", "signed_zero", "sparse", "few", "none", "nonfinite", "magnitude"]
BOOST_IM_END = ("gauss", "half", "unit", "nonfinite")
SHAPES = [("fast", 4096, None), ("main", 4097, S2PRO_MAIN), ("fast", 64, None), ("main", 65, TINY_MAIN),
          ("fast", 4352, None), ("fast", 1, None)]


def _oracle_draws(L, E, T, top_p, ids, masked):
    out, pinned = [], []
    for r in range(L.shape[0]):
        row = L[r].copy()
        if masked is not None:
            row[masked] = -np.inf
        tok, diag = oracle.draw(row, T, top_p, 30, E[r], ids)
        out.append(tok)
        pinned.append(tok < 0 or (float(diag[1]) > 1e-5 and float(diag[2]) - float(diag[3]) > 1e-5))
    return np.asarray(out), np.asarray(pinned)


@pytest.mark.parametrize("T,top_p", [(0.7, 0.85), (1.0, 0.93)])
@pytest.mark.parametrize("kind", KINDS)
def test_draw_matches_oracle(kind, T, top_p):
    import dual_ar_tts_gb300 as pkg
    rng = np.random.default_rng(1000 * KINDS.index(kind) + int(round(T * 10)))
    compared = total = 0
    for role, n, ids_of in SHAPES:
        L = _rows(kind, n, rng)
        if role == "main" and kind in BOOST_IM_END:
            # im_end the largest logit of its row: masking it changes the draw
            fin = np.where(np.isfinite(L[:, :n - 1]), L[:, :n - 1], -np.inf)
            L[:, n - 1] = fin.max(axis=1) + 1.0
        E = (-np.log(rng.uniform(1e-6, 1.0, (ROWS, 30)))).astype(np.float32)
        dl, de = torch.from_numpy(L).cuda(), torch.from_numpy(E).cuda()
        for block_end in ([False, True] if role == "main" else [False]):
            if role == "main":
                ids = np.concatenate([ids_of["sem_begin"] + np.arange(n - 1), [ids_of["im_end"]]]).astype(np.int32)
                got = pkg.draw(dl, de, T, top_p, ids_of["sem_begin"], ids_of["im_end"], block_end).cpu().numpy()
            else:
                ids = None
                got = pkg.draw(dl, de, T, top_p).cpu().numpy()
            want, pinned = _oracle_draws(L, E, T, top_p, ids, n - 1 if block_end else None)
            torch.cuda.synchronize()
            for r in np.flatnonzero(pinned):
                assert int(got[r]) == int(want[r]), (kind, role, n, block_end, int(r), int(got[r]), int(want[r]))
            if block_end:
                assert not np.any(got == ids_of["im_end"]), "a masked im_end was drawn"
            compared += int(pinned.sum())
            total += len(pinned)
    print(kind, T, top_p, f"compared {compared} of {total} rows")
    assert compared >= 0.9 * total
