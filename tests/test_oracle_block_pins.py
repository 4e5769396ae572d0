"""Pins of the oracle's transformer block composition to closed forms.

The block is described the same way for the Slow-AR and the Fast-AR transformer (s2.cpp analysis
ch.02 "Overall architecture and Dual-AR data flow" §3.2; ch.06 "Fast-AR codebook decoding and the
generation main loop" §3: fused wqkv, view split into q / k / v, per-head q/k RMSNorm, then RoPE,
GQA attention, output projection with residual, RMSNorm, SwiGLU feed-forward with residual;
Mizuoto "Fish Speech" engine page, "how it works" and "numerics").

Each test runs the oracle on a micro model (dim 4, two query heads sharing one KV head, head_dim 2,
FFN 2, one layer, fp32, eps 0, RoPE table not rounded) whose weights are chosen by hand so that
the expected result is a short closed form written out below with scalars and 2-vectors in
float64.  With head_dim 2 the single RoPE pair has frequency base^0 = 1, so position p rotates by
p radians.  The observables are the K/V rows the block stores in the cache, the final-norm hidden
of the last position (final norm weights 1 and eps 0, so it is the residual's direction) and the
fast_norm rows of a Fast-AR call.

Each pin is chosen so that one plausible misreading of the composition fails it:
* the SwiGLU gate on w3 instead of w1, or one matrix for both;
* k and v (or q and k) rows of wqkv swapped in the split;
* the q/k RMSNorm applied after RoPE instead of before (invisible with unit norm weights);
* RoPE applied to v, a missing 1/sqrt(head_dim) score scale;
* the feed-forward norm taken from the block input instead of the post-attention residual.
"""
import math

import numpy as np

import oracle

D, HQ, HKV, HD, FF = 4, 2, 1, 2, 2
QKV = (HQ + 2 * HKV) * HD

MICRO = dict(
    dim=D, n_layer=1, n_head=HQ, n_kv_head=HKV, head_dim=HD, ffn=FF, vocab=16,
    sem_begin=8, sem_end=11, im_end=12, n_codebooks=2, codebook_size=4,
    sem_scale=1.0, norm_eps=0.0, rope_base=1e6, qk_norm=1, rope_table_bf16=0,
    fast_dim=D, fast_n_layer=1, fast_n_head=HQ, fast_n_kv_head=HKV, fast_head_dim=HD,
    fast_ffn=FF, fast_window=3, has_fast_project_in=0,
    weight_dtype=0, kv_dtype=0, weight_fp8=0,
)

# residual inputs (text ids 1 and 2: the input is embeddings[id], sem_scale 1, no codebook term)
X0 = np.array([1.0, -1.0, 1.0, -1.0])   # rms 1
X1 = np.array([1.0, 1.0, -1.0, -1.0])   # rms 1


def _layer(wqkv=None, qn=(1.0, 1.0), kn=(1.0, 1.0), wo=None, w1=None, w3=None, w2=None):
    z = lambda *s: np.zeros(s, np.float32)
    return [np.ones(D, np.float32),
            z(QKV, D) if wqkv is None else np.float32(wqkv),
            np.float32(qn), np.float32(kn),
            z(D, HQ * HD) if wo is None else np.float32(wo),
            np.ones(D, np.float32),
            z(FF, D) if w1 is None else np.float32(w1),
            z(FF, D) if w3 is None else np.float32(w3),
            z(D, FF) if w2 is None else np.float32(w2)]


def _weights(layer, fast_layer=None, fe=None):
    E = np.zeros((MICRO["vocab"], D), np.float32)
    E[1], E[2] = X0, X1
    CE = np.zeros((2 * 4, D), np.float32)
    FE = np.zeros((4, D), np.float32) if fe is None else np.float32(fe)
    w = [E, CE, np.ones(D, np.float32)] + layer
    w += [None, FE, np.ones(D, np.float32), np.zeros((4, D), np.float32)]
    w += fast_layer if fast_layer is not None else _layer()
    return w


def _prompt(*ids):
    return np.array([[i, 0, 0] for i in ids], np.int32)


def _dir(v):
    v = np.asarray(v, np.float64)
    return v / math.sqrt(np.mean(v * v))


def _rot(v, ang):
    c, s = math.cos(ang), math.sin(ang)
    return np.array([v[0] * c - v[1] * s, v[0] * s + v[1] * c])


def _silu(a):
    return a / (1.0 + math.exp(-a))


# wqkv rows: q head 0 (rows 0-1), q head 1 (rows 2-3), k (rows 4-5), v (rows 6-7)
WQKV = np.array([
    [1.0, 0.0, 0.0, 0.0],     # q0 = (x_0, x_1)
    [0.0, 1.0, 0.0, 0.0],
    [0.0, 0.0, 0.5, 0.0],     # q1 = (0.5 x_2, -x_3)
    [0.0, 0.0, 0.0, -1.0],
    [0.0, 3.0, 0.0, 0.0],     # k = (3 x_1, x_3)
    [0.0, 0.0, 0.0, 1.0],
    [0.5, 0.0, 0.0, 0.0],     # v = (0.5 x_0, 0.25 x_2)
    [0.0, 0.0, 0.25, 0.0],
])
QN, KN = (0.5, 3.0), (2.0, 0.5)


def _qkv(x):
    y = WQKV @ x
    return y[0:2], y[2:4], y[4:6], y[6:8]


def _normed(v, w):
    """per-head RMSNorm of a 2-vector (eps 0) times its weight"""
    v = np.asarray(v, np.float64)
    return v / math.sqrt(np.mean(v * v)) * np.asarray(w)


def test_block_swiglu_gate_is_w1():
    # one position, attention contributes nothing (wo = 0); the FFN input is x0 itself (rms 1)
    w1 = [[1, 0, 0, 0], [0, 0, 0, 0]]      # w1·h = (1, 0)
    w3 = [[2, 0, 0, 0], [0, 0, 0, 0]]      # w3·h = (2, 0)
    w2 = [[1, 0], [0, 0], [0, 0], [0, 0]]
    s = oracle.Session(MICRO, _weights(_layer(wqkv=WQKV, w1=w1, w3=w3, w2=w2)), 4)
    _, hidden = s.prefill(_prompt(1))
    # x' = x0 + w2·(silu(w1 h) ⊙ w3 h) = x0 + (2 silu(1), 0, 0, 0)
    exp = X0 + np.array([2.0 * _silu(1.0), 0, 0, 0])
    np.testing.assert_allclose(hidden, _dir(exp), rtol=1e-6, atol=1e-7)
    # the reading with the gate on w3 gives a different direction
    assert np.max(np.abs(_dir(X0 + [_silu(2.0), 0, 0, 0]) - _dir(exp))) > 1e-2


def test_block_wqkv_split_and_cache_rows_at_position_zero():
    s = oracle.Session(MICRO, _weights(_layer(wqkv=WQKV, qn=QN, kn=KN)), 4)
    s.prefill(_prompt(1))
    k, v = s.kv(0, 0, 1)
    q0, q1, kk, vv = _qkv(X0)
    # slot 0: k normalised with k_norm (RoPE at position 0 is the identity), v as projected
    np.testing.assert_allclose(k[0, 0], _normed(kk, KN), rtol=1e-6)
    np.testing.assert_allclose(v[0, 0], vv, rtol=1e-6)
    np.testing.assert_allclose(k[0, 0], [-2.0 * 3 / math.sqrt(5), -0.5 / math.sqrt(5)], rtol=1e-6)
    np.testing.assert_allclose(v[0, 0], [0.5, 0.25], rtol=1e-6)


def test_block_single_position_attention_returns_v_through_wo():
    # one position: softmax over one slot is 1, so each head's output is v; wo = identity
    s = oracle.Session(MICRO, _weights(_layer(wqkv=WQKV, qn=QN, kn=KN, wo=np.eye(4))), 4)
    _, hidden = s.prefill(_prompt(1))
    _, _, _, vv = _qkv(X0)
    exp = X0 + np.concatenate([vv, vv])        # both query heads read the one KV head
    np.testing.assert_allclose(hidden, _dir(exp), rtol=1e-6, atol=1e-7)


def test_block_norm_before_rope_in_the_cache_at_position_one():
    s = oracle.Session(MICRO, _weights(_layer(wqkv=WQKV, qn=QN, kn=KN)), 4)
    s.prefill(_prompt(1, 2))
    k, v = s.kv(0, 0, 2)
    _, _, kk, vv = _qkv(X1)
    exp_k = _rot(_normed(kk, KN), 1.0)            # norm, weight, then rotate by 1 rad
    np.testing.assert_allclose(k[1, 0], exp_k, rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(v[1, 0], vv, rtol=1e-6)   # v is not rotated
    wrong = _normed(_rot(kk, 1.0), KN)             # rotate, then norm: a different vector
    assert np.max(np.abs(wrong - exp_k)) > 1e-2


def _two_position_residual(x0, x1):
    """x1 + wo·o1 for the second position with wo = identity (closed form, head_dim 2)."""
    _, _, k0, v0 = _qkv(x0)
    q0, q1, k1, v1 = _qkv(x1)
    ks = [_normed(k0, KN), _rot(_normed(k1, KN), 1.0)]
    vs = [v0, v1]
    out = []
    for q in (q0, q1):
        qr = _rot(_normed(q, QN), 1.0)
        sc = np.array([qr @ kj for kj in ks]) / math.sqrt(HD)
        p = np.exp(sc - sc.max())
        p /= p.sum()
        out.append(p[0] * vs[0] + p[1] * vs[1])
    return x1 + np.concatenate(out)


def test_block_two_positions_q_norm_rope_scale_and_causal_attention():
    s = oracle.Session(MICRO, _weights(_layer(wqkv=WQKV, qn=QN, kn=KN, wo=np.eye(4))), 4)
    _, hidden = s.prefill(_prompt(1, 2))
    exp = _two_position_residual(X0, X1)
    np.testing.assert_allclose(hidden, _dir(exp), rtol=2e-6, atol=1e-6)


def test_block_ffn_reads_the_post_attention_residual():
    w1 = [[1, 0, 0, 0], [0, 0, 0, 0]]
    w3 = [[2, 0, 0, 0], [0, 0, 0, 0]]
    w2 = [[1, 0], [0, 0], [0, 0], [0, 0]]
    s = oracle.Session(MICRO, _weights(_layer(wqkv=WQKV, qn=QN, kn=KN, wo=np.eye(4), w1=w1, w3=w3, w2=w2)), 4)
    _, hidden = s.prefill(_prompt(1))
    _, _, _, vv = _qkv(X0)
    xm = X0 + np.concatenate([vv, vv])              # (1.5, -0.75, 1.5, -0.75)
    h0 = xm[0] / math.sqrt(np.mean(xm * xm))        # ffn_norm(x_mid)_0 (weights 1)
    exp = xm + np.array([_silu(h0) * 2.0 * h0, 0, 0, 0])
    np.testing.assert_allclose(hidden, _dir(exp), rtol=1e-6, atol=1e-7)
    # a parallel block (FFN on the block input x0) would give another direction
    par = xm + np.array([_silu(1.0) * 2.0, 0, 0, 0])
    assert np.max(np.abs(_dir(par) - _dir(exp))) > 1e-2


def test_fast_block_same_composition():
    # Fast-AR call with one prefix code: row 0 = the hidden itself (no fast_project_in), row 1 =
    # fast_embeddings[code]; positions 0 and 1 from zero; fast_norm weights 1
    fe = np.zeros((4, D))
    fe[3] = X1
    w = _weights(_layer(), fast_layer=_layer(wqkv=WQKV, qn=QN, kn=KN, wo=np.eye(4)), fe=fe)
    s = oracle.Session(MICRO, w, 4)
    _, rows = s.fast_logits(X0.astype(np.float32), [3], rows=True)
    _, _, _, v0 = _qkv(X0)
    np.testing.assert_allclose(rows[0], _dir(X0 + np.concatenate([v0, v0])), rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(rows[1], _dir(_two_position_residual(X0, X1)), rtol=2e-6, atol=1e-6)
