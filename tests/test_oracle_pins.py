"""Pins of the CPU oracle to facts fixed by the pages and by mathematics (closed forms,
invariants, special cases, brute force, statistics) — never to the oracle itself.

Sources: s2.cpp analysis ch.02 "Overall architecture and Dual-AR data flow" (§2 dims, §3.1
token layout, §3.2 embedding sum and tied logits, §3.4 feedback), ch.06 "Fast-AR codebook
decoding and the generation main loop" (§1-§4 Fast-AR, §5 sem_mask / loop, §5.2 clamp, §5.3
min_tokens_before_end, §6 RAS, §8 compaction), Mizuoto "Fish Speech" engine page (RMSNorm in
fp32, adjacent-pair RoPE with a bf16 table, top-k 30, argmax(probs / -log u), draw order,
repeat_interleave of K/V).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synth

TINY = synth.CONFIGS["tiny"]["dims"]


def _bf16(x):
    return torch.tensor(np.float32(x)).to(torch.bfloat16).float().item()


# ------------------------------------------------------------------ RMSNorm

def test_rmsnorm_closed_forms():
    # x = [3, 4]: mean square 12.5
    out = oracle.rmsnorm([3.0, 4.0], eps=1e-6)
    np.testing.assert_allclose(out, np.array([3, 4]) / math.sqrt(12.5 + 1e-6), rtol=1e-6)
    # eps sits inside the square root: x = [1e-3, 1e-3], eps = 1e-6 -> 1e-3 / sqrt(2e-6)
    out = oracle.rmsnorm([1e-3, 1e-3], eps=1e-6)
    np.testing.assert_allclose(out, [1e-3 / math.sqrt(2e-6)] * 2, rtol=1e-6)
    # constant vector -> sign(a)·w
    w = np.array([0.5, 2.0, -1.0, 3.0], np.float32)
    out = oracle.rmsnorm(np.full(4, -7.0), w=w, eps=0.0)
    np.testing.assert_allclose(out, -w, rtol=1e-6)


def test_rmsnorm_scale_invariance():
    x = synth.normal_f32(5, 1, 257)
    np.testing.assert_allclose(oracle.rmsnorm(x * 1000.0, eps=0.0), oracle.rmsnorm(x, eps=0.0), rtol=2e-6, atol=1e-7)


# --------------------------------------------------------------------- RoPE

def test_rope_position_zero_is_identity():
    x = synth.normal_f32(1, 2, 128)
    np.testing.assert_array_equal(oracle.rope(x, 0), x)


def test_rope_adjacent_pairs_and_frequencies():
    # hd = 4: pair (0,1) has theta_0 = 1, pair (2,3) theta_1 = base^(-1/2) = 1e-3 at base 1e6
    out = oracle.rope([1.0, 0.0, 0.0, 0.0], 1, base=1e6, table_bf16=False)
    np.testing.assert_allclose(out, [math.cos(1), math.sin(1), 0, 0], rtol=1e-6, atol=1e-7)
    out = oracle.rope([0.0, 0.0, 1.0, 0.0], 1000, base=1e6, table_bf16=False)
    np.testing.assert_allclose(out, [0, 0, math.cos(1), math.sin(1)], rtol=1e-6, atol=1e-6)
    # second component of a pair: (0, 1) -> (-sin, cos)
    out = oracle.rope([0.0, 1.0], 2, base=1e6, table_bf16=False)
    np.testing.assert_allclose(out, [-math.sin(2), math.cos(2)], rtol=1e-6)


def test_rope_table_rounded_to_bf16():
    out = oracle.rope([1.0, 0.0], 3, base=1e6, table_bf16=True)
    np.testing.assert_array_equal(out, np.float32([_bf16(math.cos(3)), _bf16(math.sin(3))]))


def test_rope_norm_and_relative_position():
    rng = np.random.default_rng(0)
    q, k = rng.standard_normal(64).astype(np.float32), rng.standard_normal(64).astype(np.float32)
    rq = oracle.rope(q, 37, table_bf16=False)
    np.testing.assert_allclose(np.hypot(rq[0::2], rq[1::2]), np.hypot(q[0::2], q[1::2]), rtol=1e-5)
    a = float(np.dot(oracle.rope(q, 37, table_bf16=False), oracle.rope(k, 30, table_bf16=False)))
    b = float(np.dot(oracle.rope(q, 1037, table_bf16=False), oracle.rope(k, 1030, table_bf16=False)))
    assert abs(a - b) < 2e-3 * (1 + abs(a))


# ---------------------------------------------------------------- attention

def test_attention_single_slot_returns_value():
    rng = np.random.default_rng(1)
    q = rng.standard_normal((2, 8)).astype(np.float32)
    K = rng.standard_normal((2, 1, 8)).astype(np.float32)
    V = rng.standard_normal((2, 1, 8)).astype(np.float32)
    np.testing.assert_allclose(oracle.attention(q, K, V), V[:, 0, :], rtol=1e-6)


def test_attention_two_slot_closed_form():
    # scores·scale = [0, ln 3] -> weights [1/4, 3/4]; scale = 1/sqrt(hd) with hd = 4
    hd = 4
    q = np.zeros((1, hd), np.float32)
    q[0, 0] = 1.0
    K = np.zeros((1, 2, hd), np.float32)
    K[0, 1, 0] = math.log(3.0) * math.sqrt(hd)
    V = np.array([[[1, 2, 3, 4], [5, 6, 7, 8]]], np.float32)
    np.testing.assert_allclose(oracle.attention(q, K, V)[0], 0.25 * V[0, 0] + 0.75 * V[0, 1], rtol=1e-6)


def test_attention_uniform_keys_give_mean_value():
    rng = np.random.default_rng(2)
    q = rng.standard_normal((4, 8)).astype(np.float32)
    K = np.repeat(rng.standard_normal((2, 1, 8)).astype(np.float32), 6, axis=1)
    V = rng.standard_normal((2, 6, 8)).astype(np.float32)
    out = oracle.attention(q, K, V)
    exp = np.repeat(V.mean(axis=1), 2, axis=0)
    np.testing.assert_allclose(out, exp, rtol=1e-5, atol=1e-6)


def test_attention_brute_force_fp64_and_causal_prefix():
    rng = np.random.default_rng(3)
    hq, hkv, hd, S = 4, 2, 8, 6
    q = rng.standard_normal((hq, hd)).astype(np.float32)
    K = rng.standard_normal((hkv, S, hd)).astype(np.float32)
    V = rng.standard_normal((hkv, S, hd)).astype(np.float32)
    for n in range(1, S + 1):
        out = oracle.attention(q, K, V, n=n)
        for h in range(hq):
            g = h // (hq // hkv)
            s = [sum(float(q[h, e]) * float(K[g, j, e]) for e in range(hd)) / math.sqrt(hd) for j in range(n)]
            m = max(s)
            p = [math.exp(v - m) for v in s]
            z = sum(p)
            o = [sum(p[j] / z * float(V[g, j, e]) for j in range(n)) for e in range(hd)]
            np.testing.assert_allclose(out[h], o, rtol=1e-5, atol=1e-6)


def test_gqa_equals_mha_on_repeat_interleaved_kv():
    rng = np.random.default_rng(4)
    hq, hkv, hd, S = 8, 2, 16, 5
    q = rng.standard_normal((hq, hd)).astype(np.float32)
    K = rng.standard_normal((hkv, S, hd)).astype(np.float32)
    V = rng.standard_normal((hkv, S, hd)).astype(np.float32)
    gqa = oracle.attention(q, K, V)
    mha = oracle.attention(q, np.repeat(K, hq // hkv, axis=0), np.repeat(V, hq // hkv, axis=0))
    np.testing.assert_array_equal(gqa, mha)
    np.testing.assert_array_equal(oracle.gqa_head_map(32, 8), np.repeat(np.arange(8), 4))


def test_attention_slot_permutation_invariance():
    rng = np.random.default_rng(5)
    q = rng.standard_normal((2, 8)).astype(np.float32)
    K = rng.standard_normal((1, 7, 8)).astype(np.float32)
    V = rng.standard_normal((1, 7, 8)).astype(np.float32)
    perm = rng.permutation(7)
    np.testing.assert_allclose(oracle.attention(q, K, V), oracle.attention(q, K[:, perm], V[:, perm]), rtol=1e-5,
                               atol=1e-6)


# ---------------------------------------------------------- embedding sum

def _tiny_weights(zero_out=(), seed=0, jitter=0.0):
    w = synth.make_weights(TINY, seed, norm_jitter=jitter)
    specs = synth.weight_specs(TINY)
    for i, (name, _, _) in enumerate(specs):
        if any(name.endswith(z) for z in zero_out):
            w[i] = np.zeros_like(w[i])
    return w


def test_embed_closed_forms():
    d = TINY
    w = _tiny_weights()
    E, CE = w[0], w[1]
    s = oracle.Session(d, w, 8)
    # semantic position: sem_scale·E[r0] + Σ_c CE[c·CBS + code_c]
    vals = [d["sem_begin"] + 3, 5, 0, 63, 17]
    exp = np.float32(d["sem_scale"]) * E[vals[0]]
    acc = np.zeros(d["dim"], np.float64)
    for c in range(d["n_codebooks"]):
        acc += CE[c * d["codebook_size"] + vals[1 + c]]
    np.testing.assert_allclose(s.embed(vals), exp + acc, rtol=1e-5, atol=1e-7)
    # text position: the codebook rows do not contribute
    t1 = s.embed([17, 5, 0, 63, 17])
    t2 = s.embed([17, 0, 0, 0, 0])
    np.testing.assert_array_equal(t1, t2)
    np.testing.assert_allclose(t1, np.float32(d["sem_scale"]) * E[17], rtol=1e-6)


def test_embed_codebook_offset_uses_codebook_index():
    d = dict(TINY)
    w = _tiny_weights()
    CE = np.zeros_like(w[1])
    marker_row = 2 * d["codebook_size"] + 9      # codebook 2 (matrix row 3), code 9
    CE[marker_row, 0] = 1.0
    w[1] = CE
    s = oracle.Session(d, w, 8)
    sem = d["sem_begin"]
    assert s.embed([sem, 0, 0, 9, 0])[0] - np.float32(d["sem_scale"]) * w[0][sem, 0] == pytest.approx(1.0)
    for other in ([sem, 9, 0, 0, 0], [sem, 0, 9, 0, 0], [sem, 0, 0, 0, 9], [sem, 0, 0, 8, 0]):
        assert s.embed(other)[0] == pytest.approx(np.float32(d["sem_scale"]) * w[0][sem, 0])


# ---------------------------------------------------------------- sem_mask

def test_sem_mask_admissible_set():
    for d in (TINY, synth.CONFIGS["frame"]["dims"]):
        m = oracle.sem_mask(d, False)
        fin = set(np.flatnonzero(np.isfinite(m)).tolist())
        assert fin == set(range(d["sem_begin"], d["sem_end"] + 1)) | {d["im_end"]}
        assert len(fin) == d["codebook_size"] + 1
        m2 = oracle.sem_mask(d, True)
        assert np.isfinite(m2).sum() == d["codebook_size"] and not np.isfinite(m2[d["im_end"]])
    assert len(oracle.admissible_ids(synth.CONFIGS["frame"]["dims"])) == 4097


# ---------------------------------------------------------------- sampler

def _E(vals):
    e = np.ones(30, np.float32)
    e[:len(vals)] = vals
    return e


def test_draw_dominant_logit_always_wins():
    lg = np.zeros(100, np.float32)
    lg[42] = 100.0
    for seed in range(20):
        E = synth.exponential_f32(seed, 9, 30)
        assert oracle.draw(lg, 0.8, 0.8, 30, E)[0] == 42


def test_draw_equal_variates_give_argmax():
    rng = np.random.default_rng(6)
    for _ in range(20):
        lg = rng.standard_normal(300).astype(np.float32)
        assert oracle.draw(lg, 0.8, 0.95, 30, np.ones(30, np.float32))[0] == int(np.argmax(lg))


def test_draw_equal_logits_top_p_cut_and_argmin_variate():
    # 50 equal logits: ranks are ids 0..29 (ties -> lower id); π_r = 1/30;
    # top_p = 0.81 keeps ranks r with r/30 < 0.81 -> ranks 0..24
    lg = np.zeros(50, np.float32)
    E = np.linspace(2.0, 1.0, 30).astype(np.float32)     # smallest variate at rank 29
    assert oracle.draw(lg, 1.0, 0.81, 30, E)[0] == 24     # best kept rank is the last kept one
    assert oracle.draw(lg, 1.0, 1.0, 30, E)[0] == 29      # all 30 kept
    E2 = E.copy()
    E2[7] = 0.01
    assert oracle.draw(lg, 1.0, 0.81, 30, E2)[0] == 7


def test_draw_never_beyond_top_k():
    lg = np.linspace(1.0, 0.0, 40).astype(np.float32)    # ids 30..39 are ranks >= 30
    E = np.full(30, 1.0, np.float32)
    for seed in range(50):
        E = synth.exponential_f32(seed, 11, 30)
        tok, _ = oracle.draw(lg, 1.0, 1.0, 30, E)
        assert 0 <= tok < 30


def test_draw_top_p_zero_gives_argmax():
    rng = np.random.default_rng(7)
    lg = rng.standard_normal(500).astype(np.float32)
    for seed in range(20):
        assert oracle.draw(lg, 0.8, 1e-9, 30, synth.exponential_f32(seed, 12, 30))[0] == int(np.argmax(lg))


def test_draw_ties_go_to_lower_id():
    lg = np.full(10, -np.inf, np.float32)
    lg[7] = lg[3] = 0.5
    assert oracle.draw(lg, 1.0, 1.0, 30, np.ones(30, np.float32))[0] == 3


def test_draw_masked_entries_ignored_and_ids_mapping():
    lg = np.array([0.1, 0.9, 0.3], np.float32)
    ids = np.array([500, 20, 7], np.int32)
    assert oracle.draw(lg, 1.0, 1e-9, 30, np.ones(30, np.float32), ids=ids)[0] == 20
    lg = np.array([-np.inf, 0.2, -np.inf], np.float32)
    assert oracle.draw(lg, 1.0, 0.5, 30, np.ones(30, np.float32))[0] == 1


@pytest.mark.parametrize("temp,logits,probs", [
    (1.0, np.log([0.5, 0.3, 0.2]), [0.5, 0.3, 0.2]),
    (0.5, np.array([0.0, math.log(2.0), -np.inf]), [0.2, 0.8, 0.0]),   # z = [0, 2 ln 2]: π ∝ [1, 4]
])
def test_draw_is_a_sample_from_softmax_chi_square(temp, logits, probs):
    n = 100_000
    lg = np.asarray(logits, np.float32)
    E = synth.exponential_f32(123, 77, n * 30).reshape(n, 30)
    counts = np.zeros(3)
    for i in range(n):
        counts[oracle.draw(lg, temp, 1.0, 30, E[i])[0]] += 1
    p = np.asarray(probs)
    for c, pi in zip(counts, p):
        sd = math.sqrt(n * pi * (1 - pi)) + 1e-9
        assert abs(c - n * pi) < 4.5 * sd + (1 if pi == 0 else 0)


# ----------------------------------------------------- the frame loop logic

class _FakeSession:
    """Stands in for the model: fixed logits / hidden, so that a test can script the draws."""

    def __init__(self, d):
        self.d = d
        self.steps = []

    def fast_logits(self, hidden, prefix):
        return np.zeros(self.d["codebook_size"], np.float32)

    def step(self, vals):
        self.steps.append(list(vals))
        return np.zeros(self.d["vocab"], np.float32), np.zeros(self.d["dim"], np.float32)


def _script(d, d0s, d1s, codes=None):
    f = np.zeros((len(d0s), 11), np.int32)
    for i, (a, b) in enumerate(zip(d0s, d1s)):
        f[i, 0], f[i, 1] = a, b
        f[i, 2:2 + d["n_codebooks"] - 1] = (codes or [i % d["codebook_size"]] * 10)[:d["n_codebooks"] - 1]
    return f


def _run_scripted(d, d0s, d1s, min_tokens=0):
    fs = _FakeSession(d)
    n = len(d0s)
    expo = np.ones((n, 11, 30), np.float32)
    s = synth.sampling("tiny", min_tokens_before_end=min_tokens)
    lg = np.zeros(d["vocab"], np.float32)
    res = oracle.run_frames(fs, lg, np.zeros(d["dim"], np.float32), n, s, expo,
                            forced=_script(d, d0s, d1s), trace=False)
    return res, fs


def test_ras_trigger_within_window_and_not_beyond():
    d = TINY
    S = d["sem_begin"]
    red = S + 60
    # frame 2 repeats frame 0's token (distance 2) -> replaced by the redraw
    res, _ = _run_scripted(d, [S + 1, S + 2, S + 1], [red] * 3)
    assert res["tokens"] == [S + 1, S + 2, red]
    # a repeat at distance 11 is outside the 10-token window -> kept
    d0s = [S + i for i in range(11)] + [S + 0]
    res, _ = _run_scripted(d, d0s, [red] * 12)
    assert res["tokens"][-1] == S + 0
    # distance 10 -> still inside
    d0s = [S + i for i in range(10)] + [S + 0]
    res, _ = _run_scripted(d, d0s, [red] * 11)
    assert res["tokens"][-1] == red
    # the window holds final tokens: the replacement is what later frames compare against
    res, _ = _run_scripted(d, [S + 1, S + 1, S + 9], [S + 5, S + 9, S + 7])
    assert res["tokens"] == [S + 1, S + 9, S + 7]


def test_im_end_stops_and_is_never_emitted():
    d = TINY
    S = d["sem_begin"]
    res, fs = _run_scripted(d, [S + 1, S + 2, d["im_end"], S + 3], [S] * 4)
    assert res["stopped"] and len(res["codes"]) == 2 and len(fs.steps) == 2


def test_redraw_may_yield_im_end_and_frame_proceeds():
    d = TINY
    S = d["sem_begin"]
    res, fs = _run_scripted(d, [S + 1, S + 1], [S + 2, d["im_end"]])
    assert res["tokens"] == [S + 1, d["im_end"]]
    assert res["codes"][1][0] == d["codebook_size"] - 1           # 4160 - 4096 clamps to 63
    assert fs.steps[1][0] == d["im_end"]


def test_sem_code_clamp():
    d = synth.CONFIGS["frame"]["dims"]
    assert oracle.sem_code(d["sem_begin"] + 5, d) == 5
    assert oracle.sem_code(d["sem_end"], d) == 4095
    assert oracle.sem_code(d["im_end"], d) == 0                    # 151645 < sem_begin
    assert oracle.sem_code(d["sem_end"] + 40, d) == 4095


def test_compaction_layout_with_early_stop():
    d = TINY
    S = d["sem_begin"]
    fs = _FakeSession(d)
    forced = _script(d, [S + 1, S + 2, S + 3, d["im_end"]], [S] * 4)
    forced[:, 2:5] = [[11, 12, 13], [21, 22, 23], [31, 32, 33], [0, 0, 0]]
    res = oracle.run_frames(fs, np.zeros(d["vocab"], np.float32), np.zeros(d["dim"], np.float32), 4,
                            synth.sampling("tiny", min_tokens_before_end=0), np.ones((4, 11, 30), np.float32),
                            forced=forced, trace=False)
    n = 3
    flat = res["flat"]
    assert flat.size == 4 * n
    assert list(flat[0:n]) == [1, 2, 3]                              # codebook 0 = sem_code
    assert list(flat[n:2 * n]) == [11, 21, 31]
    assert list(flat[3 * n:4 * n]) == [13, 23, 33]
    # the fed-back step input is [token, code_0..code_{NCB-1}]
    assert fs.steps[0] == [S + 1, 1, 11, 12, 13]


def test_min_tokens_before_end_masks_im_end():
    d = TINY
    fs = _FakeSession(d)
    lg = np.full(d["vocab"], -5.0, np.float32)
    lg[d["im_end"]] = 50.0                                            # im_end would win whenever allowed
    s = synth.sampling("tiny", min_tokens_before_end=3)

    class _S(_FakeSession):
        def step(self, vals):
            super().step(vals)
            return lg.copy(), np.zeros(d["dim"], np.float32)
    fs = _S(d)
    res = oracle.run_frames(fs, lg.copy(), np.zeros(d["dim"], np.float32), 10, s, np.ones((10, 11, 30), np.float32),
                            trace=False)
    assert res["stopped"] and len(res["codes"]) == 3


# ------------------------------------------------ whole-model special cases

def test_zero_output_projections_reduce_model_to_embedding_and_tied_logits():
    d = TINY
    w = _tiny_weights(zero_out=("attention.wo", "feed_forward.w2"), jitter=0.1)
    s = oracle.Session(d, w, 40)
    p = synth.prompt("tiny")
    logits, hidden = s.prefill(p)
    x = s.embed(p[-1])
    normw = w[2].astype(np.float64)
    exp_h = x / np.sqrt(np.mean(x.astype(np.float64) ** 2) + 1e-6) * normw
    np.testing.assert_allclose(hidden, exp_h, rtol=2e-5, atol=1e-6)
    np.testing.assert_allclose(logits, w[0].astype(np.float64) @ hidden.astype(np.float64), rtol=1e-4, atol=1e-5)
    # Fast-AR: the last row is fast_norm(fast_embeddings[last prefix code]); row 0 is
    # fast_norm(fast_project_in · hidden); logits = fast_output · last row
    specs = [n for n, _, _ in synth.weight_specs(d)]
    P, FE, fn, FO = (w[specs.index(k)].astype(np.float64) for k in
                     ("fast_project_in", "fast_embeddings", "fast_norm", "fast_output"))
    lg, rows = s.fast_logits(hidden, [5, 9], rows=True)

    def rn(v):
        return v / np.sqrt(np.mean(v ** 2) + 1e-6) * fn
    np.testing.assert_allclose(rows[-1], rn(FE[9]), rtol=2e-5, atol=1e-6)
    np.testing.assert_allclose(rows[1], rn(FE[5]), rtol=2e-5, atol=1e-6)
    np.testing.assert_allclose(rows[0], rn(P @ hidden.astype(np.float64)), rtol=2e-4, atol=1e-5)
    np.testing.assert_allclose(lg, FO @ rows[-1].astype(np.float64), rtol=1e-4, atol=1e-6)


def test_tied_logits_brute_force():
    d = TINY
    w = _tiny_weights(jitter=0.1)
    s = oracle.Session(d, w, 40)
    logits, hidden = s.prefill(synth.prompt("tiny"))
    np.testing.assert_allclose(logits, w[0].astype(np.float64) @ hidden.astype(np.float64), rtol=1e-4, atol=1e-5)


def test_incremental_step_equals_longer_prefill():
    d = TINY
    w = _tiny_weights(jitter=0.1)
    p = synth.prompt("tiny")
    a = oracle.Session(d, w, 40)
    a.prefill(p[:-3])
    for t in range(3):
        la, ha = a.step(p[len(p) - 3 + t])
    b = oracle.Session(d, w, 40)
    lb, hb = b.prefill(p)
    np.testing.assert_allclose(la, lb, rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(ha, hb, rtol=1e-5, atol=1e-6)
    ka, va = a.kv(2, 0, 32)
    kb, vb = b.kv(2, 0, 32)
    np.testing.assert_allclose(ka, kb, rtol=1e-5, atol=1e-6)


def test_prompt_in_pieces_equals_one_prefill():
    # causal attention over every earlier slot: running the prompt in pieces changes nothing
    d = TINY
    w = _tiny_weights(jitter=0.1)
    p = synth.prompt("tiny")
    a = oracle.Session(d, w, 40)
    la, ha = a.prefill(p)
    b = oracle.Session(d, w, 40)
    lb, hb = b.prefill_chunked(p, chunk=7)
    np.testing.assert_allclose(lb, la, rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(hb, ha, rtol=1e-5, atol=1e-6)
    assert b.pos == a.pos == len(p)
    for layer in (0, d["n_layer"] - 1):
        np.testing.assert_allclose(b.kv(layer, 0, len(p))[0], a.kv(layer, 0, len(p))[0], rtol=1e-5, atol=1e-6)


def test_fast_prefix_consistency():
    d = TINY
    w = _tiny_weights(jitter=0.1)
    s = oracle.Session(d, w, 4)
    h = synth.normal_f32(3, 3, d["dim"])
    prefix = [7, 40, 2]
    _, full = s.fast_logits(h, prefix, rows=True)
    for k in range(1, len(prefix) + 1):
        _, part = s.fast_logits(h, prefix[:k], rows=True)
        np.testing.assert_allclose(part[-1], full[k], rtol=1e-5, atol=1e-6)
        np.testing.assert_allclose(part, full[:k + 1], rtol=1e-5, atol=1e-6)


def test_fast_entry_checks():
    d = TINY
    s = oracle.Session(d, _tiny_weights(), 4)
    h = np.zeros(d["dim"], np.float32)
    with pytest.raises(ValueError):
        s.fast_logits(h, [1, 2, 3, 4])        # prefix must be shorter than the codebook count
    with pytest.raises(ValueError):
        s.fast_logits(h, [64])                # code out of range


def test_fp16_kv_cache_rounds_on_store():
    d16 = dict(TINY, kv_dtype=synth.F16)
    w = _tiny_weights(jitter=0.1)
    a = oracle.Session(TINY, w, 40)
    b = oracle.Session(d16, w, 40)
    p = synth.prompt("tiny")
    a.prefill(p)
    b.prefill(p)
    k32, v32 = a.kv(0, 0, 32)          # layer 0 depends on each position's own input only
    k16, v16 = b.kv(0, 0, 32)
    np.testing.assert_array_equal(k16, k32.astype(np.float16).astype(np.float32))
    np.testing.assert_array_equal(v16, v32.astype(np.float16).astype(np.float32))


# ------------------------------------------------ stream state without a prompt

def test_kv_set_f16_widens_bit_patterns_exactly():
    d16 = dict(TINY, kv_dtype=synth.F16)
    s = oracle.Session(d16, _tiny_weights(), 8)
    H, hd = d16["n_kv_head"], d16["head_dim"]
    pats = np.array([0x3C00, 0xC000, 0x0001, 0x7BFF, 0x8000, 0x3555, 0x0400, 0xFBFF], np.uint16)
    want = np.array([1.0, -2.0, 2.0 ** -24, 65504.0, -0.0, 0.333251953125, 2.0 ** -14, -65504.0], np.float32)
    k = np.tile(pats, H * 2 * hd // len(pats)).reshape(H, 2, hd)
    v = k[:, ::-1].copy()
    s.set_kv_f16(1, k, v)
    kk, vv = s.kv(1, 0, 2)                      # [slot][head][hd]
    np.testing.assert_array_equal(kk, np.tile(want, H * 2 * hd // len(want)).reshape(H, 2, hd).transpose(1, 0, 2))
    np.testing.assert_array_equal(vv[0], kk[1])


def test_head_closed_form_and_brute_force():
    d = TINY
    w = _tiny_weights(jitter=0.1)
    s = oracle.Session(d, w, 8)
    normw = w[2].astype(np.float64)
    lg, h = s.head(np.full(d["dim"], -3.0, np.float32))
    np.testing.assert_allclose(h, -normw, rtol=1e-6)          # x = a·1: RMSNorm gives sign(a)·w
    x = synth.normal_f32(5, 5, d["dim"])
    lg, h = s.head(x)
    xd = x.astype(np.float64)
    np.testing.assert_allclose(h, xd / np.sqrt(np.mean(xd ** 2) + 1e-6) * normw, rtol=2e-5, atol=1e-6)
    np.testing.assert_allclose(lg, w[0].astype(np.float64) @ h.astype(np.float64), rtol=1e-4, atol=1e-5)
    lg2, h2 = s.head(x * 7.0)                    # scale invariance of the final norm
    np.testing.assert_allclose(h2, h, rtol=1e-5, atol=1e-6)


def test_imported_state_steps_like_the_prefilled_one():
    # a stream restored from another stream's fp16 KV and position continues identically
    d16 = dict(TINY, kv_dtype=synth.F16)
    w = _tiny_weights(jitter=0.1)
    p = synth.prompt("tiny")
    a = oracle.Session(d16, w, 40)
    a.prefill(p)
    b = oracle.Session(d16, w, 40)
    L, H, hd, n = d16["n_layer"], d16["n_kv_head"], d16["head_dim"], len(p)
    for l in range(L):
        k, v = a.kv(l, 0, n)                     # [slot][head][hd], fp16 values
        k16 = k.astype(np.float16).view(np.uint16).transpose(1, 0, 2)
        v16 = v.astype(np.float16).view(np.uint16).transpose(1, 0, 2)
        b.set_kv_f16(l, k16, v16)
    b.set_pos(n)
    vals = p[-1].copy()
    vals[0] = d16["sem_begin"] + 3
    la, ha = a.step(vals)
    lb, hb = b.step(vals)
    np.testing.assert_array_equal(la, lb)
    np.testing.assert_array_equal(ha, hb)


def test_draw_diag_reports_the_winner_rank_gap():
    # three candidates with z = 3, 2.5, 2.4 (T = 1); variates make rank 1 win
    lg = np.array([3.0, 2.5, 2.4, -5.0], np.float32)
    E = np.full(30, 100.0, np.float32)
    E[1] = 1e-3
    tok, diag = oracle.draw(lg, 1.0, 1.0, 30, E)
    assert tok == 1 and int(diag[5]) == 1
    assert abs(float(diag[6]) - 0.1) < 1e-6        # min(3 - 2.5, 2.5 - 2.4)
    tok, diag = oracle.draw(np.array([3.0], np.float32), 1.0, 1.0, 30, E)
    assert np.isinf(diag[6])


# ------------------------------------------------------------ codec front

def test_codec_latent_constant_rows_sum_closed_form():
    ncb, cbs, dim, n = 4, 64, 16, 5
    qs = [np.full((cbs, dim), np.float32(cb + 1)).view(np.uint32) >> 16 for cb in range(ncb)]
    qs = [q.astype(np.uint16) for q in qs]
    codes = synth.uniform_int(1, 2, ncb * n, 0, cbs - 1)
    lat = oracle.codec_latent(qs, codes, n)
    np.testing.assert_array_equal(lat, np.full((n, dim), ncb * (ncb + 1) / 2, np.float32))


def test_codec_latent_reads_codes_by_codebook_row():
    # codebook cb holds its row index in element cb: latent[f][cb] must be code(cb, f), read from
    # codes[cb * n_frames + f]
    ncb, cbs, dim, n = 4, 64, 8, 6
    qs = []
    for cb in range(ncb):
        q = np.zeros((cbs, dim), np.float32)
        q[:, cb] = np.arange(cbs, dtype=np.float32)
        qs.append((q.view(np.uint32) >> 16).astype(np.uint16))
    codes = synth.uniform_int(3, 4, ncb * n, 0, cbs - 1)
    lat = oracle.codec_latent(qs, codes, n)
    for cb in range(ncb):
        np.testing.assert_array_equal(lat[:, cb], codes[cb * n:(cb + 1) * n].astype(np.float32))
    np.testing.assert_array_equal(lat[:, ncb:], 0)
