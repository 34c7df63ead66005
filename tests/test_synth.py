"""The seeded input generator: published SplitMix64 outputs, storage rounding
against library casts, counter-based regeneration and the workload recipe's
distributions."""
import json
import os

import numpy as np
import torch

from transformer_layer_decode_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_splitmix64_published_outputs():
    g = json.load(open(os.path.join(GOLDEN, "splitmix64.json")))
    gamma = 0x9E3779B97F4A7C15
    got = [synth.lib().synth_splitmix64((i * gamma) % 2**64) for i in range(3)]
    assert got == [int(h, 16) for h in g["state0_outputs"]]


def test_rounding_matches_library_casts():
    rng = np.random.default_rng(5)
    x = rng.normal(0, 2, 4000).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([synth.lib().synth_round_bf16(float(v)) for v in x], np.uint16)
    assert np.array_equal(got, ref)
    y = np.concatenate([rng.normal(0, 0.002, 3000), rng.normal(0, 1e-5, 1000)]).astype(np.float32)
    ref16 = y.astype(np.float16).view(np.uint16)     # numpy: RNE, subnormals included
    got16 = np.array([synth.lib().synth_round_fp16(float(v)) for v in y], np.uint16)
    assert np.array_equal(got16, ref16)


def test_counter_based_regeneration():
    a = synth.normal_bf16(0, 3, synth.T_WQ, 0, 1000, 0.0, 0.02)
    b = synth.normal_bf16(0, 3, synth.T_WQ, 600, 400, 0.0, 0.02)
    assert np.array_equal(a[600:], b)
    c = synth.normal_bf16(0, 4, synth.T_WQ, 0, 1000, 0.0, 0.02)
    assert not np.array_equal(a, c)


def test_workload_distributions():
    w = synth.WORKLOADS["layer_h512"]
    W = synth.bf16_to_f32(synth.weight_bf16(w, 0, synth.T_WGATE))
    assert abs(W.mean()) < 1e-3 and abs(W.std() - 0.02) < 5e-4
    n = synth.bf16_to_f32(synth.norm_bf16(w, 0, synth.T_ATTN_NORM))
    assert abs(n.mean() - 1.0) < 0.02 and abs(n.std() - 0.1) < 0.02
    K, V = synth.kv_bf16(w, 0, 127)
    assert K.shape == (2, 127, 64) and abs(synth.bf16_to_f32(V).std() - 1.0) < 0.05
    # prefix property: fewer prefilled rows are a prefix of more
    K2, _ = synth.kv_bf16(w, 0, 40)
    assert np.array_equal(K2, K[:, :40])
    q, s = synth.weight_q4(w.small(weight_fmt="q4"), 0, synth.T_WQ)
    nib = np.concatenate([q & 15, q >> 4]).astype(np.int64) - 8
    assert nib.min() == -8 and nib.max() == 7 and abs(nib.mean() + 0.5) < 0.05
    sc = synth.fp16_to_f32(s)
    assert sc.min() >= 0 and abs(sc.mean() - 0.002 * np.sqrt(2 / np.pi)) < 1e-4
    x = synth.step_input(w, 0)
    assert x.dtype == np.float32 and abs(x.std() - 1) < 0.1
    assert np.array_equal(synth.bf16_to_f32(synth.lib().synth_round_bf16(float(x[0])) * np.ones(1, np.uint16)), x[:1])
