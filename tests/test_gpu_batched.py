"""CUDA path vs oracle on the batched workloads (S2-Pro shapes, bf16 weights, fp16 KV), through
the C ABI, at their full batch, context and frame counts.

An fp32 CPU prefill of 512..4096 (serving) or 30000 (long context) positions at S2-Pro width
does not finish in seconds, so each stream's decode state comes from ``s2_stream_import``:
seeded synthetic fp16 K/V for every layer and position (``synth.kv_state``; the streams of a
workload share one master state of the longest context, each taking its own prefix length) and
the stream's own last residual.  The oracle is given the same state (``Session.import_state``).

* serving (32 streams, contexts 512..4096, 128 frames): the first frames of four sampled
  streams, teacher-forced with the oracle's draws (the other streams forced with seeded
  tokens), are compared with the oracle — logits and hidden at max-abs-rel <= 2e-2, pinned
  draws and emitted codes exactly.  Then all 128 frames free-running: every frame produced,
  codes in range, the same codes on a second run, and a sub-batch decoded alone gives the
  same codes as inside the full batch.
* long context (8 streams x 30000 positions, 256 frames): the same comparison for two streams,
  then the 256 free-running frames with the same properties.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.parity import compare_frames

pytestmark = pytest.mark.gpu
TOL = 2e-2
N_CHECK = 3          # frames compared with the oracle per sampled stream


def _x_last(seed, stream, d):
    return synth.kv_state(seed, stream, dict(d, n_layer=1, n_kv_head=1), 1)[2]


def _decoder(pkg, d, dev, n, slots, lengths, kd, vd, seed):
    dec = pkg.Decoder(d, dev, max_streams=n, kv_slots=slots)
    for i, L in enumerate(lengths):
        x = torch.from_numpy(_x_last(seed, i, d)).cuda()
        dec.import_stream(i, kd[:, :, :L].contiguous(), vd[:, :, :L].contiguous(), x)
    torch.cuda.synchronize()
    return dec


def _forced_filler(seed, i, n_frames, d):
    f = np.zeros((n_frames, 11), np.int32)
    f[:, 0:2] = synth.uniform_int(seed, 5_000_000 + i, n_frames * 2, d["sem_begin"], d["sem_end"]).reshape(-1, 2)
    f[:, 2:] = synth.uniform_int(seed, 5_100_000 + i, n_frames * 9, 0, d["codebook_size"] - 1).reshape(-1, 9)
    return f


def _oracle_ref(d, host, k16, v16, L, x, n_frames, s, expo, slots):
    sess = oracle.Session(d, host, slots)
    logits, hidden = sess.import_state(k16[:, :, :L], v16[:, :, :L], x)
    ref = oracle.run_frames(sess, logits, hidden, n_frames, s, expo)
    sess.close()
    return ref


def _run_workload(pkg, s2pro, cfg_name, sampled):
    d, host, dev, names = s2pro
    cfg = synth.CONFIGS[cfg_name]
    n, K, slots, seed = cfg["streams"], cfg["frames"], cfg["kv_slots"], cfg["input_seed"]
    lengths = synth.prompt_lengths(cfg_name)
    k16, v16, _ = synth.kv_state(seed, 0, d, max(lengths))
    kd = torch.from_numpy(k16.view(np.int16)).cuda().view(torch.float16)
    vd = torch.from_numpy(v16.view(np.int16)).cuda().view(torch.float16)
    s = synth.sampling(cfg_name)

    # 1. teacher-forced first frames of the whole batch; sampled streams against the oracle
    expo = np.stack([synth.expo(seed, i, N_CHECK) for i in range(n)])
    forced = np.stack([_forced_filler(seed, i, N_CHECK, d) for i in range(n)])
    refs = {}
    for i in sampled:
        ref = _oracle_ref(d, host, k16, v16, lengths[i], _x_last(seed, i, d), N_CHECK, s, expo[i],
                          lengths[i] + N_CHECK + 1)
        assert len(ref["codes"]) == N_CHECK
        forced[i] = np.asarray(ref["draws"], np.int32)
        refs[i] = ref
    dec = _decoder(pkg, d, dev, n, slots, lengths, kd, vd, seed)
    out = dec.decode(N_CHECK, s, torch.from_numpy(expo).cuda(), torch.from_numpy(forced).cuda(), taps=True)
    assert dec.sync_status() == pkg.S2_OK, pkg.s2_last_error(dec.ctx)
    for i in sampled:
        st = compare_frames(refs[i], out, d, s, TOL, stream=i)
        print(f"{cfg_name} stream {i} (context {lengths[i]}):", st)
    assert (out["n_out"].cpu().numpy() == N_CHECK).all()
    dec.close()

    # 2. all frames free-running, twice from the same state; a sub-batch alone
    expo_d = torch.from_numpy(np.stack([synth.expo(seed, i, K) for i in range(n)])).cuda()
    runs = []
    for _ in range(2):
        dec = _decoder(pkg, d, dev, n, slots, lengths, kd, vd, seed)
        o = dec.decode(K, s, expo_d, taps=False)
        assert dec.sync_status() == pkg.S2_OK, pkg.s2_last_error(dec.ctx)
        runs.append({k: v.cpu() for k, v in o.items()})
        dec.close()
    a, b = runs
    assert (a["n_out"].numpy() == K).all()
    codes = a["codes"].numpy().reshape(n, d["n_codebooks"], K)
    assert (codes >= 0).all() and (codes < d["codebook_size"]).all()
    assert torch.equal(a["codes"], b["codes"])
    sub = list(sampled[:2])
    dec = _decoder(pkg, d, dev, n, slots, lengths, kd, vd, seed)
    o = dec.decode(K, s, expo_d[sub], stream_ids=sub, taps=False)
    assert dec.sync_status() == pkg.S2_OK, pkg.s2_last_error(dec.ctx)
    for j, i in enumerate(sub):
        assert torch.equal(o["codes"][j].cpu(), a["codes"][i]), f"stream {i} differs inside the full batch"
    dec.close()
    del kd, vd
    torch.cuda.empty_cache()


def test_serving_32_streams(s2pro):
    import dual_ar_tts_gb300 as pkg
    _run_workload(pkg, s2pro, "serving", sampled=[0, 9, 21, 31])


def test_long_context_8_streams_30000_positions(s2pro):
    import dual_ar_tts_gb300 as pkg
    _run_workload(pkg, s2pro, "longctx", sampled=[0, 7])


def test_import_rejects_bad_arguments(s2pro):
    import dual_ar_tts_gb300 as pkg
    d, host, dev, names = s2pro
    dec = pkg.Decoder(d, dev, max_streams=2, kv_slots=64)
    k = torch.zeros((d["n_layer"], d["n_kv_head"], 65, d["head_dim"]), dtype=torch.float16, device="cuda")
    x = torch.zeros(d["dim"], device="cuda")
    with pytest.raises(pkg.S2Error) as e:
        dec.import_stream(0, k, k, x)
    assert e.value.code == pkg.S2_ECAPACITY
    with pytest.raises(pkg.S2Error) as e:
        dec.import_stream(2, k[:, :, :8].contiguous(), k[:, :, :8].contiguous(), x)
    assert e.value.code == pkg.S2_EINVAL
    dec.close()


def test_mini_batched_prefill_and_frames_match_oracle():
    # three streams of a small bf16 model (4 query heads per KV head) from real prompts of
    # different lengths, decoded together, teacher-forced with the oracle's draws
    import dual_ar_tts_gb300 as pkg
    d = synth.MINI
    host = synth.make_weights(d, 7, norm_jitter=0.1)
    dev = pkg.upload_weights(host)
    prompts = [synth.make_prompt(d, 7, i, 20 + 3 * i, 6 + i) for i in range(3)]
    s = synth.sampling("tiny")
    n_frames = 6
    expo = np.stack([synth.expo(7, i, n_frames) for i in range(3)])
    refs, forced = [], np.zeros((3, n_frames, 11), np.int32)
    for i, p in enumerate(prompts):
        sess = oracle.Session(d, host, len(p) + n_frames + 1)
        ref = oracle.generate(sess, p, n_frames, s, expo[i])
        forced[i, :len(ref["draws"])] = np.asarray(ref["draws"], np.int32)
        refs.append(ref)
        sess.close()
    dec = pkg.Decoder(d, dev, max_streams=4, kv_slots=64)
    dec.prefill(prompts)
    out = dec.decode(n_frames, s, torch.from_numpy(expo).cuda(), torch.from_numpy(forced).cuda(), taps=True)
    assert dec.sync_status() == pkg.S2_OK, pkg.s2_last_error(dec.ctx)
    for i in range(3):
        st = compare_frames(refs[i], out, d, s, TOL, stream=i)
        print(f"mini stream {i}:", st)
    dec.close()


def _mini(pkg):
    d = synth.MINI
    host = synth.make_weights(d, 7, norm_jitter=0.1)
    return d, host, pkg.upload_weights(host)


def test_stop_request_and_progress():
    # frame-level cancel (ch.06 §7): a stop request ends a stream at its next frame boundary; the
    # others continue; progress reports the frames emitted; a new prefill clears the request
    import dual_ar_tts_gb300 as pkg
    d, host, dev = _mini(pkg)
    s = synth.sampling("tiny", min_tokens_before_end=100)
    prompts = [synth.make_prompt(d, 7, i, 20, 6) for i in range(3)]
    for n in (3, 1):  # batched kernels, then the single-stream kernel
        dec = pkg.Decoder(d, dev, max_streams=4, kv_slots=64)
        dec.prefill(prompts[:n])
        ex = lambda f0, k: torch.from_numpy(np.stack([synth.expo(7, i, k, f0) for i in range(n)])).cuda()
        out = dec.decode(2, s, ex(0, 2))
        assert dec.sync_status() == pkg.S2_OK
        dec.stop(n - 1)
        out = dec.decode(3, s, ex(2, 3))
        assert dec.sync_status() == pkg.S2_OK
        got = out["n_out"].cpu().numpy().tolist()
        assert got == [3] * (n - 1) + [0], got
        assert dec.progress(list(range(n))).tolist() == got
        dec.prefill([prompts[n - 1]], stream_ids=[n - 1])
        out = dec.decode(2, s, ex(0, 2)[n - 1:n], stream_ids=[n - 1])
        assert dec.sync_status() == pkg.S2_OK and int(out["n_out"][0]) == 2
        dec.close()


def test_continuous_batching_matches_each_request_decoded_alone():
    # five requests through two slots, decoded in short calls with slots refilled as requests
    # finish; each request's codes equal those of the same request decoded beside a fixed partner
    import dual_ar_tts_gb300 as pkg
    d, host, dev = _mini(pkg)
    s = synth.sampling("tiny", min_tokens_before_end=100)
    lengths = [5, 9, 3, 7, 6]
    reqs = [(synth.make_prompt(d, 7, i, 18 + 2 * i, 5 + i), lengths[i]) for i in range(5)]
    expo_fn = lambda r, f0, n: synth.expo(70 + r, 0, n, f0)
    dec = pkg.Decoder(d, dev, max_streams=2, kv_slots=64)
    got = pkg.serve(dec, reqs, slots=2, frames_per_call=2, sampling=s, expo_fn=expo_fn)
    assert dec.sync_status() == pkg.S2_OK
    dec.close()
    partner = synth.make_prompt(d, 7, 9, 16, 4)
    for r, (prompt, n) in enumerate(reqs):
        ref = pkg.Decoder(d, dev, max_streams=2, kv_slots=64)
        ref.prefill([prompt, partner])
        ex = torch.from_numpy(np.stack([expo_fn(r, 0, n), synth.expo(99, 0, n)])).cuda()
        out = ref.decode(n, s, ex)
        assert ref.sync_status() == pkg.S2_OK
        want = out["codes"][0].cpu().numpy().reshape(d["n_codebooks"], n)
        assert got[r].shape == want.shape and np.array_equal(got[r], want), r
        ref.close()
