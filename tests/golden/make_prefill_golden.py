"""Writes the oracle's outputs for long prompts into tests/golden/*.npz.

An fp32 CPU prefill of thousands of positions at S2-Pro width takes minutes to tens of minutes,
too long for a test run, so the oracle runs once here and the GPU tests compare with what it
wrote.  Only the oracle (``oracle/``) and the seeded input generators (``synth/``) are called.

Cases (the prompts are the workloads' own: 3/4 text ids, then reference positions with semantic
ids and codes; s2.cpp analysis ch.02 §3.1 token layout):

* ``serving_s12``  serving stream 12, the shortest prompt (568 positions), full S2-Pro shapes
* ``serving_s3``   serving stream 3, 2077 positions, full S2-Pro shapes
* ``longctx_s0_2l`` long-context stream 0 (30000 positions: 1000 text ids then 29000 reference
  positions), S2-Pro widths with 2 Slow-AR layers

For each: the prompt is prefilled (in pieces of 256 positions, which gives the same result as one
prefill), then 2 frames are decoded with the workload's sampler settings and the stream's own
exponential variates.  Stored: the prefill's admissible logits and hidden state, and for each
frame the draws, their diagnostics, the admissible main logits, the hidden state, the nine
Fast-AR logit vectors and the emitted codes.

    python tests/golden/make_prefill_golden.py [case ...]
"""
from __future__ import annotations

import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import synth  # noqa: E402

N_FRAMES = 2
CASES = {
    "serving_s12": dict(cfg="serving", stream=12, n_layer=None),
    "serving_s3": dict(cfg="serving", stream=3, n_layer=None),
    "longctx_s0_2l": dict(cfg="longctx", stream=0, n_layer=2),
}


def case_dims(case: dict) -> dict:
    d = synth.CONFIGS[case["cfg"]]["dims"]
    return dict(d, n_layer=case["n_layer"]) if case["n_layer"] is not None else dict(d)


def case_inputs(case: dict):
    """prompt, sampling settings and variates of a case (shared with the GPU test)"""
    cfg = synth.CONFIGS[case["cfg"]]
    prompt = synth.prompt(case["cfg"], stream=case["stream"])
    s = synth.sampling(case["cfg"])
    expo = synth.expo(cfg["input_seed"], case["stream"], N_FRAMES)
    return prompt, s, expo


def path(name: str) -> str:
    return os.path.join(HERE, f"prefill_{name}.npz")


def make(name: str) -> None:
    case = CASES[name]
    d = case_dims(case)
    prompt, s, expo = case_inputs(case)
    t0 = time.time()
    w = synth.make_weights(d, 0)
    sess = oracle.Session(d, w, len(prompt) + N_FRAMES + 1)
    logits, hidden = sess.prefill_chunked(prompt, 256)
    t1 = time.time()
    ref = oracle.run_frames(sess, logits, hidden, N_FRAMES, s, expo)
    assert len(ref["codes"]) == N_FRAMES, "the golden cases decode every frame"
    adm = oracle.admissible_ids(d)
    np.savez(path(name),
             prompt_len=np.int32(len(prompt)), n_layer=np.int32(d["n_layer"]), stream=np.int32(case["stream"]),
             prefill_logits=logits[adm].astype(np.float32), prefill_hidden=hidden.astype(np.float32),
             draws=np.asarray(ref["draws"], np.int32), diags=np.asarray(ref["diags"], np.float64),
             main_logits=np.stack(ref["main_logits"]).astype(np.float32),
             hidden=np.stack(ref["hidden"]).astype(np.float32),
             fast_logits=np.stack(ref["fast_logits"]).astype(np.float32),
             codes=np.asarray(ref["codes"], np.int32), flat=np.asarray(ref["flat"], np.int32))
    print(f"{name}: {len(prompt)} positions x {d['n_layer']} layers, prefill {t1 - t0:.0f} s, "
          f"frames {time.time() - t1:.0f} s -> {path(name)}", flush=True)


def load(name: str) -> dict:
    """The stored outputs in the shape oracle.run_frames returns them (for tests.parity)."""
    z = np.load(path(name))
    ref = {k: z[k] for k in z.files}
    ref["main_logits"] = list(ref["main_logits"])
    ref["hidden"] = list(ref["hidden"])
    ref["fast_logits"] = list(ref["fast_logits"])
    ref["draws"] = [list(map(int, r)) for r in ref["draws"]]
    ref["codes"] = [list(map(int, r)) for r in ref["codes"]]
    return ref


if __name__ == "__main__":
    for n in (sys.argv[1:] or list(CASES)):
        make(n)
