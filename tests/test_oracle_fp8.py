"""Pins of the oracle's e4m3 weight quantisation (low-precision weight streaming).

The format is the OCP 8-bit float E4M3 (sign, 4 exponent bits with bias 7, 3 mantissa bits, no
infinities, S.1111.111 = NaN, subnormals m*2^-9, largest finite 448); the library rounds to
nearest with ties to the even mantissa and saturates at 448, with one fp32 scale per row
(max|row| / 448).  The oracle's code is pinned to things other than itself:

* every code's value against torch's float8_e4m3fn (a library decoding);
* encoding against torch's float -> float8_e4m3fn conversion on values inside the range, and
  against a brute-force search over the 254 finite values (nearest, ties to the even code) on
  random values and on the exact midpoints between neighbours;
* closed-form cases: ties at 1, in the subnormal range and at the top; saturation;
* the quantiser's invariants (the largest element of a row maps to +-448 exactly, the error is
  within half a step, zero rows) and the binding: a session reading e4m3 codes gives the same
  numbers as one given the dequantised fp32 matrices.
"""
import numpy as np
import pytest

import oracle
import synth

FINITE = [c for c in range(256) if (c & 0x7F) != 0x7F]


def _torch():
    return pytest.importorskip("torch")


def test_code_values_match_torch_float8():
    torch = _torch()
    codes = torch.tensor(FINITE, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_value(c) for c in FINITE])
    assert np.array_equal(np.signbit(got), np.signbit(ref))
    assert np.array_equal(got, ref)
    assert oracle.e4m3_value(0x7E) == 448.0 and oracle.e4m3_value(0x01) == 2.0 ** -9


def test_every_code_round_trips():
    for c in FINITE:
        assert oracle.e4m3_encode(np.float32(oracle.e4m3_value(c))) == c, hex(c)


def _brute(x):
    """Nearest finite e4m3 value by search; ties to the code with an even last bit; |x| >= 448 -> 448."""
    if abs(x) >= 448.0:
        return 0x7E | (0x80 if np.signbit(x) else 0)
    best, bd = None, None
    for c in FINITE:
        v = oracle.e4m3_value(c)
        if np.signbit(v) != np.signbit(x):
            continue
        dist = abs(float(x) - v)
        if bd is None or dist < bd or (dist == bd and (c & 1) == 0 and (best & 1) == 1):
            best, bd = c, dist
    return best


def test_encode_matches_brute_force_and_midpoints():
    rng = np.random.default_rng(5)
    xs = list(rng.normal(0, 30, 300).astype(np.float32))
    xs += list((rng.uniform(-1, 1, 200) * 2.0 ** rng.integers(-14, 9, 200)).astype(np.float32))
    pos = sorted(oracle.e4m3_value(c) for c in FINITE if c < 0x80)
    mids = [np.float32((a + b) / 2) for a, b in zip(pos[:-1], pos[1:])]  # exact in fp32
    xs += mids + [-m for m in mids]
    for x in xs:
        assert oracle.e4m3_encode(x) == _brute(float(x)), (x, hex(oracle.e4m3_encode(x)))


def test_encode_matches_torch_conversion_in_range():
    torch = _torch()
    rng = np.random.default_rng(6)
    x = np.concatenate([rng.normal(0, 40, 4000), rng.uniform(-1, 1, 4000) * 2.0 ** rng.integers(-16, 8, 4000)])
    x = x.astype(np.float32)
    x = x[np.abs(x) < 448]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(v) for v in x], np.uint8)
    assert np.array_equal(got, ref)


def test_closed_form_cases():
    enc = oracle.e4m3_encode
    assert enc(1.0) == 0x38
    assert enc(1.0625) == 0x38          # midway 1 and 1.125: even mantissa 000
    assert enc(1.1875) == 0x3A          # midway 1.125 and 1.25: even mantissa 010
    assert enc(2.0 ** -10) == 0x00      # half the smallest subnormal: ties to zero
    assert enc(3 * 2.0 ** -10) == 0x02  # midway 2^-9 and 2^-8: even m = 2
    assert enc(15 * 2.0 ** -10) == 0x08  # midway 7*2^-9 and 2^-6: the smallest normal
    assert enc(448.0) == 0x7E and enc(464.0) == 0x7E and enc(1e30) == 0x7E
    assert enc(-1e30) == 0xFE and enc(-0.0) == 0x80 and enc(0.0) == 0x00
    assert enc(240.0) == 0x77 and enc(-2.0 ** -6) == 0x88


def test_quantiser_invariants():
    rng = np.random.default_rng(7)
    w32 = rng.normal(0, 0.02, (40, 256)).astype(np.float32)
    w32[3] = 0.0
    w32[4, :] = 0.0
    w32[4, 17] = -3.5
    w32[5] *= 1e-30                     # tiny row: scale far below 1
    w = (w32.view(np.uint32) >> 16).astype(np.uint16)  # truncation to bf16 patterns is fine here
    codes, scales = oracle.quant_e4m3(w)
    wf = (w.astype(np.uint32) << 16).view(np.float32)
    vals = np.vectorize(oracle.e4m3_value)(codes)
    amax = np.abs(wf).max(axis=1)
    assert np.array_equal(scales, (amax / np.float32(448)).astype(np.float32))
    assert np.all((codes & 0x7F) != 0x7F)
    for r in range(w.shape[0]):
        if amax[r] == 0:
            assert scales[r] == 0 and not codes[r].any()
            continue
        k = int(np.argmax(np.abs(wf[r])))
        assert abs(vals[r, k]) == 448.0
        deq = vals[r] * np.float64(scales[r])
        bound = np.maximum(np.abs(wf[r]) * 2.0 ** -4, 2.0 ** -10 * scales[r]) * (1 + 1e-6)
        assert np.all(np.abs(deq - wf[r]) <= bound), r
    assert codes[4, 17] == 0xFE and np.count_nonzero(codes[4]) == 1


def test_session_reading_codes_equals_dequantised_fp32_weights():
    d = synth.MINI
    host = synth.make_weights(d, 3, norm_jitter=0.1)
    quant = oracle.quantize_projections(d, host)
    assert sorted(quant) == sorted(oracle.projection_indices(d))
    deq = []
    for i, w in enumerate(host):
        if w is None:
            deq.append(None)
        elif i in quant:
            c, s = quant[i]
            v = np.vectorize(oracle.e4m3_value)(c) * s.astype(np.float64)[:, None]
            deq.append(v.astype(np.float32).reshape(w.shape))
        else:
            deq.append((w.astype(np.uint32) << 16).view(np.float32))
    prompt = synth.make_prompt(d, 3, 0, 12, 4)
    a = oracle.Session(d, host, 32, quant=quant)
    b = oracle.Session(dict(d, weight_dtype=synth.F32), deq, 32)
    la, ha = a.prefill(prompt)
    lb, hb = b.prefill(prompt)
    assert np.array_equal(la, lb) and np.array_equal(ha, hb)
    # and the e4m3 model is a different model from the bf16 one (the codes are in use)
    c = oracle.Session(d, host, 32)
    lc, _ = c.prefill(prompt)
    assert not np.array_equal(la, lc)
    assert np.max(np.abs(la - lc)) < 0.1 * np.max(np.abs(lc))
    for s in (a, b, c):
        s.close()


@pytest.mark.parametrize("cfg", ["frame", "tiny"])
def test_projection_indices_name_exactly_the_projection_matrices(cfg):
    # the table indices the oracle reads as e4m3 are the projections, by the weight table's names
    d = synth.CONFIGS[cfg]["dims"]
    specs = synth.weight_specs(d)
    idx = oracle.projection_indices(d)
    want = {i for i, (name, shape, _) in enumerate(specs)
            if name.split(".")[-1] in ("wqkv", "wo", "w1", "w3", "w2")
            or (name == "fast_project_in" and d["has_fast_project_in"]) or name == "fast_output"}
    assert sorted(idx) == sorted(want) and len(idx) == len(set(idx))
    assert len(idx) == 5 * (d["n_layer"] + d["fast_n_layer"]) + 1 + int(bool(d["has_fast_project_in"]))
    assert all(len(specs[i][1]) == 2 for i in idx)
