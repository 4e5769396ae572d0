"""fp8 e4m3 weight streaming on the GPU, through the C ABI, against the oracle.

* the quantisation (codes and row scales) equals the oracle's bit for bit on seeded bf16
  matrices and on rows built to hit the edge cases (zero rows, signed zeros, subnormal codes,
  ties, the largest and smallest bf16 magnitudes, a ragged column count);
* the projection kernel's fp8 expansion passed its check against the hardware conversion (a
  context with weight_fp8 = 1 initialises only when it does);
* a small bf16 model decoded with fp8 projections, three streams together and one stream alone,
  teacher-forced with the oracle's draws: the oracle reads the same e4m3 codes and scales
  (logits and hidden at max-abs-rel <= 2e-2, pinned draws and codes exactly);
* S2-Pro, one stream: a 512-position prompt through the fp8 prompt projections and frames with a
  batch of one, against the oracle;
* the S2-Pro serving workload with fp8 projections: two sampled streams of the 32 against the
  oracle for their first frames, then free-running frames decoded twice with the same codes.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.parity import compare_frames

pytestmark = pytest.mark.gpu
TOL = 2e-2


def _bf16(a32):
    """fp32 -> bf16 bit patterns, round to nearest even."""
    u = np.ascontiguousarray(a32, np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def _dev_bf16(w16):
    return torch.from_numpy(w16.view(np.int16)).cuda().view(torch.bfloat16)


def test_quantisation_bit_exact():
    import dual_ar_tts_gb300 as pkg
    rng = np.random.default_rng(11)
    for rows, cols in ((300, 2560), (7, 77), (1, 9728)):
        w = synth.normal_bf16(11, rows * 7 + cols, rows * cols, 0.0, 0.02).reshape(rows, cols)
        if rows >= 7:
            w = w.copy()
            w[0] = 0                                     # zero row
            w[1] = 0x8000                                # negative zeros only
            w[2] = _bf16(rng.normal(0, 1, cols) * 1e-36)  # tiny magnitudes (bf16 subnormals too)
            w[3] = _bf16(rng.normal(0, 1, cols) * 1e37)   # huge magnitudes
            w[4] = _bf16(np.where(np.arange(cols) % 2 == 0, 1.0, 1.0 / 448 * 2.0 ** -9 * 1.5))  # subnormal ties
            w[5] = _bf16(rng.uniform(-1, 1, cols) * 2.0 ** rng.integers(-20, 1, cols))  # wide dynamic range
            w[6, :] = _bf16(np.float32(448.0))
        codes, scales = pkg.quantize_e4m3(_dev_bf16(w))
        rc, rs = oracle.quant_e4m3(w)
        assert np.array_equal(scales.cpu().numpy().view(np.uint32), rs.view(np.uint32)), (rows, cols)
        got = codes.cpu().numpy()
        bad = np.argwhere(got != rc)
        assert bad.size == 0, (rows, cols, bad[:5], got[tuple(bad[0])] if bad.size else None)


def test_quantise_rejects_bad_arguments():
    import dual_ar_tts_gb300 as pkg
    w = torch.zeros((4, 8), dtype=torch.bfloat16, device="cuda")
    c = torch.empty((4, 8), dtype=torch.uint8, device="cuda")
    s = torch.empty(4, dtype=torch.float32, device="cuda")
    with pytest.raises(pkg.S2Error) as e:
        pkg.s2_quantize_e4m3(w.data_ptr(), 0, 8, c.data_ptr(), s.data_ptr())
    assert e.value.code == pkg.S2_EINVAL
    with pytest.raises(pkg.S2Error):
        pkg.s2_quantize_e4m3(w.data_ptr(), 4, 8, c.data_ptr(), s.data_ptr() + 1)


def _mini_run(pkg, n_streams, n_frames, seed=7):
    d = synth.MINI
    host = synth.make_weights(d, seed, norm_jitter=0.1)
    dev = pkg.upload_weights(host)
    quant = oracle.quantize_projections(d, host)
    prompts = [synth.make_prompt(d, seed, i, 20 + 3 * i, 6 + i) for i in range(n_streams)]
    s = synth.sampling("tiny")
    expo = np.stack([synth.expo(seed, i, n_frames) for i in range(n_streams)])
    refs, forced = [], np.zeros((n_streams, n_frames, 11), np.int32)
    for i, p in enumerate(prompts):
        sess = oracle.Session(d, host, len(p) + n_frames + 1, quant=quant)
        ref = oracle.generate(sess, p, n_frames, s, expo[i])
        forced[i, :len(ref["draws"])] = np.asarray(ref["draws"], np.int32)
        refs.append(ref)
        sess.close()
    dec = pkg.Decoder(dict(d, weight_fp8=1), dev, max_streams=4, kv_slots=64)
    dec.prefill(prompts)
    out = dec.decode(n_frames, s, torch.from_numpy(expo).cuda(), torch.from_numpy(forced).cuda(), taps=True)
    assert dec.sync_status() == pkg.S2_OK, pkg.s2_last_error(dec.ctx)
    for i in range(n_streams):
        st = compare_frames(refs[i], out, d, s, TOL, stream=i)
        print(f"mini fp8 stream {i} of {n_streams}:", st)
    dec.close()
    return host, dev, quant


def test_mini_fp8_streams_match_oracle():
    import dual_ar_tts_gb300 as pkg
    _mini_run(pkg, 3, 6)


def test_mini_fp8_single_stream_matches_oracle():
    import dual_ar_tts_gb300 as pkg
    _mini_run(pkg, 1, 6)


def test_fp8_needs_the_batched_engine_shapes():
    import dual_ar_tts_gb300 as pkg
    # bf16, lengths multiples of 128, but 2 query heads per KV head: not a batched-engine shape
    d = dict(synth.CONFIGS["tiny"]["dims"], weight_dtype=synth.BF16, kv_dtype=synth.F16, weight_fp8=1)
    host = synth.make_weights(d, 1)
    dev = pkg.upload_weights(host)
    with pytest.raises(pkg.S2Error) as e:
        pkg.Decoder(d, dev, max_streams=1, kv_slots=64)
    assert e.value.code == pkg.S2_EINVAL


def test_s2pro_fp8_serving_streams_match_oracle(s2pro):
    import dual_ar_tts_gb300 as pkg
    from tests.test_gpu_batched import _decoder, _forced_filler, _x_last
    d, host, dev, names = s2pro
    cfg = synth.CONFIGS["serving"]
    n, slots, seed = cfg["streams"], cfg["kv_slots"], cfg["input_seed"]
    lengths = synth.prompt_lengths("serving")
    k16, v16, _ = synth.kv_state(seed, 0, d, max(lengths))
    kd = torch.from_numpy(k16.view(np.int16)).cuda().view(torch.float16)
    vd = torch.from_numpy(v16.view(np.int16)).cuda().view(torch.float16)
    s = synth.sampling("serving")
    quant = oracle.quantize_projections(d, host)
    n_check, sampled = 2, [0, 21]
    expo = np.stack([synth.expo(seed, i, n_check) for i in range(n)])
    forced = np.stack([_forced_filler(seed, i, n_check, d) for i in range(n)])
    refs = {}
    for i in sampled:
        sess = oracle.Session(d, host, lengths[i] + n_check + 1, quant=quant)
        logits, hidden = sess.import_state(k16[:, :, :lengths[i]], v16[:, :, :lengths[i]], _x_last(seed, i, d))
        refs[i] = oracle.run_frames(sess, logits, hidden, n_check, s, expo[i])
        sess.close()
        forced[i] = np.asarray(refs[i]["draws"], np.int32)
    d8 = dict(d, weight_fp8=1)
    dec = _decoder(pkg, d8, dev, n, slots, lengths, kd, vd, seed)
    out = dec.decode(n_check, s, torch.from_numpy(expo).cuda(), torch.from_numpy(forced).cuda(), taps=True)
    assert dec.sync_status() == pkg.S2_OK, pkg.s2_last_error(dec.ctx)
    for i in sampled:
        st = compare_frames(refs[i], out, d, s, TOL, stream=i)
        print(f"serving fp8 stream {i} (context {lengths[i]}):", st)
    dec.close()
    K = 16
    expo_d = torch.from_numpy(np.stack([synth.expo(seed, i, K) for i in range(n)])).cuda()
    runs = []
    for _ in range(2):
        dec = _decoder(pkg, d8, dev, n, slots, lengths, kd, vd, seed)
        o = dec.decode(K, s, expo_d, taps=False)
        assert dec.sync_status() == pkg.S2_OK, pkg.s2_last_error(dec.ctx)
        runs.append(o["codes"].cpu())
        assert (o["n_out"].cpu().numpy() == K).all()
        dec.close()
    assert torch.equal(runs[0], runs[1])
    del kd, vd
    torch.cuda.empty_cache()


def test_s2pro_fp8_single_stream_prefill_and_frames_match_oracle(s2pro):
    # one stream: the 512-position prompt through the fp8 prompt projections (128-position chunks,
    # 256 MMA columns), then frames on the batched engine with a batch of one, against the oracle
    import dual_ar_tts_gb300 as pkg
    d, host, dev, names = s2pro
    cfg = synth.CONFIGS["frame"]
    n_frames = 2
    prompt = synth.prompt("frame")
    s = synth.sampling("frame")
    expo = synth.expo(cfg["input_seed"], 0, n_frames)
    quant = oracle.quantize_projections(d, host)
    sess = oracle.Session(d, host, len(prompt) + n_frames + 1, quant=quant)
    ref = oracle.generate(sess, prompt, n_frames, s, expo)
    sess.close()
    forced = np.zeros((n_frames, 11), np.int32)
    forced[:len(ref["draws"])] = np.asarray(ref["draws"], np.int32)
    dec = pkg.Decoder(dict(d, weight_fp8=1), dev, max_streams=1, kv_slots=1024)
    dec.prefill([prompt])
    out = dec.decode(n_frames, s, torch.from_numpy(expo).cuda()[None], torch.from_numpy(forced).cuda()[None],
                     taps=True)
    assert dec.sync_status() == pkg.S2_OK, pkg.s2_last_error(dec.ctx)
    st = compare_frames(ref, out, d, s, TOL)
    print("fp8 single-stream parity:", st)
    dec.close()


def test_fp8_context_refuses_fast_alone():
    import dual_ar_tts_gb300 as pkg
    d = synth.MINI
    dev = pkg.upload_weights(synth.make_weights(d, 7, norm_jitter=0.1))
    dec = pkg.Decoder(dict(d, weight_fp8=1), dev, max_streams=1, kv_slots=64)
    hidden = torch.zeros((1, d["dim"]), device="cuda")
    prefix = torch.zeros((1, d["n_codebooks"] - 1), dtype=torch.int32, device="cuda")
    with pytest.raises(pkg.S2Error) as e:
        dec.fast_logits(hidden, prefix)
    assert e.value.code == pkg.S2_ESTATE
    dec.close()
