"""CUDA path vs oracle at the decode loop's edge cases and on the serving / long-context prompts.

* min_tokens_before_end (s2.cpp analysis ch.06 "Fast-AR codebook decoding and the generation main
  loop" §5.3): im_end is masked for frame f's main draw while f < min_tokens and allowed from then
  on.  The im_end embedding row is pointed along the model's hidden states so that im_end wins as
  soon as it is allowed: the oracle and the GPU must both stop exactly at frame min_tokens,
  whether the frames run in one call or in two (the frame count carries over).  Both decode
  engines: one stream (persistent kernel) and two streams (batched kernels, per-stream limits).
* repetition-aware redraw yielding im_end (ch.06 §6: only the trigger excludes im_end): the frame
  proceeds with sem_code clamped and im_end is fed back as the next Slow-AR input (a text
  position, no codebook term); every later frame is compared with the oracle.
* continuous batching with teacher-forced draws (ch.06 §7; the serving loop of the Mizuoto page):
  requests refilled into freed slots, one stopped by im_end mid-call, one repeating a recent token
  (redraw) across a call boundary; each request's codes equal the oracle's for the same draws.
* serving and long-context prompts prefilled on the GPU from their real prompts (the shortest and a
  2077-position serving stream at S2-Pro shapes; the 30000-position long-context prompt at S2-Pro
  widths with 2 Slow-AR layers), then 2 teacher-forced frames, against oracle outputs stored by
  tests/golden/make_prefill_golden.py (an fp32 CPU prefill of these prompts takes minutes).
"""
import time

import numpy as np
import pytest
import torch

import oracle
import synth
from tests.golden import make_prefill_golden as golden
from tests.parity import compare_frames

pytestmark = pytest.mark.gpu


def _boosted(d, w, prompts, n, expo, s):
    """weights whose im_end row lies along the mean direction of the oracle's hidden states (of
    every stream's frames)"""
    H = []
    for i, prompt in enumerate(prompts):
        ref = oracle.generate(oracle.Session(d, w, len(prompt) + n + 1), prompt, n,
                              dict(s, min_tokens_before_end=n), expo[i])
        H += [h / np.linalg.norm(h) for h in np.asarray(ref["hidden"], np.float64)]
    u = np.mean(H, axis=0)
    u /= np.linalg.norm(u)
    w2 = [None if x is None else x.copy() for x in w]
    if d["weight_dtype"] == synth.BF16:
        w2[0][d["im_end"]] = (np.float32(4.0 * u).view(np.uint32) >> 16).astype(np.uint16)  # bf16 bits
    else:
        w2[0][d["im_end"]] = (4.0 * u).astype(np.float32)
    return w2


@pytest.mark.parametrize("engine", ["one_stream_f32", "two_streams_bf16"])
def test_min_tokens_boundary_stops_exactly_there(engine):
    import dual_ar_tts_gb300 as pkg
    cfg = synth.CONFIGS["tiny"]
    d = cfg["dims"] if engine == "one_stream_f32" else dict(cfg["dims"], weight_dtype=synth.BF16, kv_dtype=synth.F16)
    tol = 1e-4 if engine == "one_stream_f32" else 2e-2
    n, split = 16, 5
    n_streams = 1 if engine == "one_stream_f32" else 2
    mins = [8, 5][:n_streams]
    prompts = [synth.prompt("tiny")] + ([synth.make_prompt(d, 3, 1, 22, 7)] if n_streams == 2 else [])
    expo = np.stack([synth.expo(0, i, n) for i in range(n_streams)])
    w = _boosted(d, synth.make_weights(d, 0, norm_jitter=0.1), prompts, n, expo, synth.sampling("tiny"))
    ss = [synth.sampling("tiny", min_tokens_before_end=m) for m in mins]
    refs = []
    forced = np.zeros((n_streams, n, 11), np.int32)
    for i in range(n_streams):
        ref = oracle.generate(oracle.Session(d, w, 64), prompts[i], n, ss[i], expo[i])
        assert ref["stopped"] and len(ref["codes"]) == mins[i], (i, len(ref["codes"]))
        forced[i, :len(ref["draws"])] = np.asarray(ref["draws"], np.int32)
        refs.append(ref)
    dec = pkg.Decoder(d, pkg.upload_weights(w), max_streams=n_streams, kv_slots=64)
    dec.prefill(prompts)
    ex = torch.from_numpy(expo).cuda()
    fo = torch.from_numpy(forced).cuda()
    a = dec.decode(split, ss, ex[:, :split].contiguous(), fo[:, :split].contiguous(), taps=True)
    b = dec.decode(n - split, ss, ex[:, split:].contiguous(), fo[:, split:].contiguous(), taps=True)
    assert dec.sync_status() == pkg.S2_OK, pkg.s2_last_error(dec.ctx)
    ncb = d["n_codebooks"]
    for i in range(n_streams):
        na, nb = int(a["n_out"][i]), int(b["n_out"][i])
        assert na == min(split, mins[i]) and na + nb == mins[i], (i, na, nb)
        # the im_end draw of frame min_tokens is the GPU's own (its margin makes it pinned)
        fb = mins[i] - split
        assert int(b["draws"][i, fb, 0]) == d["im_end"], b["draws"][i, fb].tolist()
        codes = np.concatenate([a["codes"][i, :ncb * na].cpu().numpy().reshape(ncb, na),
                                b["codes"][i, :ncb * nb].cpu().numpy().reshape(ncb, nb)], axis=1)
        assert np.array_equal(codes.reshape(-1), refs[i]["flat"]), i
        # logits and draws of the frames of the second call against the oracle's
        sub = dict(refs[i])
        for k in ("main_logits", "hidden", "diags", "draws", "fast_logits", "codes"):
            sub[k] = refs[i][k][split:]
        sub["flat"] = oracle.compact(refs[i]["codes"][split:], d)
        print(engine, "stream", i, compare_frames(sub, b, d, ss[i], tol, stream=i))
    dec.close()


@pytest.mark.parametrize("engine", ["one_stream_f32", "two_streams_bf16"])
def test_redraw_yielding_im_end_is_fed_back(engine):
    import dual_ar_tts_gb300 as pkg
    cfg = synth.CONFIGS["tiny"]
    d = cfg["dims"] if engine == "one_stream_f32" else dict(cfg["dims"], weight_dtype=synth.BF16, kv_dtype=synth.F16)
    tol = 1e-4 if engine == "one_stream_f32" else 2e-2
    n, f_red = 10, 4
    n_streams = 1 if engine == "one_stream_f32" else 2
    w = synth.make_weights(d, 0, norm_jitter=0.1)
    s = synth.sampling("tiny", min_tokens_before_end=n)
    prompts = [synth.prompt("tiny")] + ([synth.make_prompt(d, 3, 1, 22, 7)] if n_streams == 2 else [])
    expo = np.stack([synth.expo(5, i, n) for i in range(n_streams)])
    forced = np.zeros((n_streams, n, 11), np.int32)
    refs = []
    for i in range(n_streams):
        free = oracle.generate(oracle.Session(d, w, 64), prompts[i], n, s, expo[i])
        fr = np.asarray(free["draws"], np.int32)
        if i == 0:
            # frame f_red repeats the previous frame's token (in the window, semantic): the redraw
            # is used, and it is forced to im_end
            fr[f_red, 0] = free["tokens"][f_red - 1]
            fr[f_red, 1] = d["im_end"]
        ref = oracle.generate(oracle.Session(d, w, 64), prompts[i], n, s, expo[i], forced=fr)
        if i == 0:
            assert ref["tokens"][f_red] == d["im_end"] and len(ref["codes"]) == n
            assert ref["codes"][f_red][0] == oracle.sem_code(d["im_end"], d) == d["codebook_size"] - 1
        forced[i] = fr  # exactly the outcomes the oracle was forced with
        refs.append(ref)
    dec = pkg.Decoder(d, pkg.upload_weights(w), max_streams=n_streams, kv_slots=64)
    dec.prefill(prompts)
    out = dec.decode(n, s, torch.from_numpy(expo).cuda(), torch.from_numpy(forced).cuda(), taps=True)
    assert dec.sync_status() == pkg.S2_OK, pkg.s2_last_error(dec.ctx)
    for i in range(n_streams):
        st = compare_frames(refs[i], out, d, s, tol, stream=i)
        print(engine, "stream", i, st)
        assert st["frames"] == n
    dec.close()


def test_continuous_batching_with_forced_draws_matches_oracle():
    import dual_ar_tts_gb300 as pkg
    d = synth.MINI
    host = synth.make_weights(d, 7, norm_jitter=0.1)
    dev = pkg.upload_weights(host)
    s = synth.sampling("tiny", min_tokens_before_end=0)
    lengths = [5, 9, 3, 7, 6]
    reqs = [(synth.make_prompt(d, 7, i, 18 + 2 * i, 5 + i), lengths[i]) for i in range(5)]
    expo_fn = lambda r, f0, n: synth.expo(70 + r, 0, n, f0)
    forced_all, want = [], []
    for r, (prompt, n) in enumerate(reqs):
        sess = oracle.Session(d, host, len(prompt) + n + 1)
        ex = expo_fn(r, 0, n)
        free = oracle.generate(sess, prompt, n, s, ex)
        fr = np.zeros((n, 11), np.int32)
        fr[:len(free["draws"])] = np.asarray(free["draws"], np.int32)
        fr[:, 0] = np.where(fr[:, 0] == d["im_end"], d["sem_begin"], fr[:, 0])
        if r == 1:
            fr[4, 0] = d["im_end"]                  # request 1 stops at frame 4, inside a call
        if r == 3:
            fr[2, 0] = free["tokens"][1]            # request 3 repeats frame 1's token at frame 2
        ref = oracle.generate(oracle.Session(d, host, len(prompt) + n + 1), prompt, n, s, ex, forced=fr)
        forced_all.append(fr)
        want.append(ref)
    assert len(want[1]["codes"]) == 4 and want[1]["stopped"]
    forced_fn = lambda r, f0, n: forced_all[r][f0:f0 + n]
    dec = pkg.Decoder(d, dev, max_streams=2, kv_slots=64)
    got = pkg.serve(dec, reqs, slots=2, frames_per_call=2, sampling=s, expo_fn=expo_fn, forced_fn=forced_fn)
    assert dec.sync_status() == pkg.S2_OK
    dec.close()
    for r in range(len(reqs)):
        ref = want[r]
        exp = np.asarray(ref["codes"], np.int32).T if ref["codes"] else np.zeros((d["n_codebooks"], 0), np.int32)
        assert got[r].shape == exp.shape and np.array_equal(got[r], exp), (r, got[r], exp)


def _subset(names_full, tensors, d_sub):
    by = dict(zip(names_full, tensors))
    return [by[n] for n, _, _ in synth.weight_specs(d_sub)]


def _golden_run(pkg, s2pro, names, tol):
    d_full, host, dev, all_names = s2pro
    refs = [golden.load(nm) for nm in names]
    cases = [golden.CASES[nm] for nm in names]
    d = golden.case_dims(cases[0])
    inputs = [golden.case_inputs(c) for c in cases]
    slots = max(len(p) for p, _, _ in inputs) + golden.N_FRAMES + 8
    dec = pkg.Decoder(d, _subset(all_names, dev, d), max_streams=len(names), kv_slots=slots)
    t0 = time.perf_counter()
    dec.prefill([p for p, _, _ in inputs])
    torch.cuda.synchronize()
    pf = time.perf_counter() - t0
    expo = torch.from_numpy(np.stack([e for _, _, e in inputs])).cuda()
    forced = torch.from_numpy(np.stack([np.asarray(r["draws"], np.int32) for r in refs])).cuda()
    out = dec.decode(golden.N_FRAMES, [s for _, s, _ in inputs], expo, forced, taps=True)
    assert dec.sync_status() == pkg.S2_OK, pkg.s2_last_error(dec.ctx)
    for i, nm in enumerate(names):
        assert int(refs[i]["prompt_len"]) == len(inputs[i][0])
        st = compare_frames(refs[i], out, d, inputs[i][1], tol, stream=i)
        print(f"{nm}: prefill of {len(inputs[i][0])} positions x {d['n_layer']} layers, {st}")
    print(f"GPU prefill of {[len(p) for p, _, _ in inputs]} positions: {pf * 1e3:.1f} ms")
    dec.close()


def test_serving_prompts_prefilled_on_the_gpu_match_oracle(s2pro):
    import dual_ar_tts_gb300 as pkg
    _golden_run(pkg, s2pro, ["serving_s12", "serving_s3"], 2e-2)


def test_longctx_prompt_prefilled_on_the_gpu_matches_oracle(s2pro):
    import dual_ar_tts_gb300 as pkg
    _golden_run(pkg, s2pro, ["longctx_s0_2l"], 2e-2)
