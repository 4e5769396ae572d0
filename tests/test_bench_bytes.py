"""The bench's algorithmic bytes per frame (the roofline's numerator) against a count made from the
weight table itself: every 2-D matrix of the table read once per use — Slow-AR layer matrices once
per frame, Fast-AR layer matrices and fast_output once per Fast-AR call (nine per frame),
fast_project_in once — plus the admissible tied-logit rows of the embedding table, the gathered
embedding rows, and the fp16 KV cache over the context.  Norm vectors (a few hundred KB) are not
counted by either side."""
import re

import pytest

import bench
import synth


def _count(d, ctx, fp8=False):
    e = 2
    ncalls = d["n_codebooks"] - 1
    total = 0
    for name, shape, is_norm in synth.weight_specs(d):
        if len(shape) != 2:
            continue
        rows, cols = shape
        size = rows * cols + 4 * rows if fp8 else rows * cols * e
        if re.match(r"layers\.\d+\.", name):
            total += size
        elif re.match(r"fast_layers\.\d+\.", name) or name == "fast_output":
            total += ncalls * size
        elif name == "fast_project_in":
            total += size
        elif name == "embeddings":
            # admissible rows for the tied logits (semantic ids + im_end) and the frame's
            # semantic-token row for the next Slow-AR input
            total += (d["codebook_size"] + 1) * cols * e + cols * e
        elif name == "codebook_embeddings":
            total += d["n_codebooks"] * cols * e  # one row per codebook of the next input
        elif name == "fast_embeddings":
            total += ncalls * cols * e  # codes 0..8 feed Fast-AR positions 1..9
        else:
            raise AssertionError(f"unclassified matrix {name}")
    kv = d["n_layer"] * d["n_kv_head"] * d["head_dim"] * 2 * 2 * (ctx + 1)
    return total + kv


@pytest.mark.parametrize("cfg", ["frame", "tiny"])
@pytest.mark.parametrize("ctx", [0, 512, 4000])
def test_frame_bytes_equal_the_weight_table_count(cfg, ctx):
    d = synth.CONFIGS[cfg]["dims"]
    got, parts = bench.frame_bytes(d, ctx)
    assert got == _count(d, ctx)
    assert sum(parts.values()) <= got


def test_frame_bytes_fp8_projections():
    d = dict(synth.CONFIGS["frame"]["dims"], weight_fp8=1)
    got, _ = bench.frame_bytes(d, 512)
    # e4m3 codes + one fp32 scale per row for the projection matrices; embedding rows stay bf16
    assert got == _count(d, 512, fp8=True)


def test_s2pro_frame_is_about_fifteen_gigabytes():
    d = synth.CONFIGS["frame"]["dims"]
    got, parts = bench.frame_bytes(d, 640)
    assert 14.8e9 < got < 14.9e9
    assert abs(parts["slow"] - 7.2666e9) < 1e6 and abs(parts["fast"] - 7.4685e9) < 1e6
