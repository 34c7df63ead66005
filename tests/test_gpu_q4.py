"""GPU parity of the int4-weight / int8-activation path.

- every layer's output against the fp64 oracle (same float tolerance);
- the integer block dots bit-exact: the GPU's own int8 GEMV inputs (activation
  tap) and the int4 weights give, in int64 on the CPU, exactly the int32 dots
  the GPU kernels computed (block-dot tap), for all four projections;
- the GPU's int8 activations against the oracle's quantisation of the same
  layer input: equal up to +-1 where fp32 and fp64 straddle a rounding boundary.
"""
import numpy as np
import pytest

from harness import (Q4_SLOTS, assert_close, oracle_stack, q4_code_flips, run_gpu, run_oracle,
                     tiled_rows_to_abi)
from oracle import oracle as orc
from transformer_layer_decode_gb300 import dec, synth, workload

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

# bounds of the integer decisions (see test_gpu_full_size)
Q4_FLIP_FRACTION = (1e-3, 5e-3, 1e-3, 1e-3)
Q4_FLIP_DISTANCE = 0.05

SMALL = {
    "q4_gqa4_d64": synth.Workload("q4_gqa4_d64", 2, 512, 8, 2, 64, 1408, prefill=100, steps=3,
                                  weight_fmt="q4"),
    "q4_mha_d128": synth.Workload("q4_mha_d128", 2, 1024, 8, 8, 128, 2816, prefill=70, steps=2,
                                  weight_fmt="q4"),
    "q4_ragged_empty": synth.Workload("q4_ragged_empty", 1, 1088, 16, 4, 64, 1216, prefill=0,
                                      steps=2, weight_fmt="q4"),
}


# fused plans: the int8 GEMV inputs quantized by every CTA of the GEMV
# (default), or published once by the kernel that produces the vector (publish;
# five- and four-kernel plans)
MODES = {
    "fused_graph": {},
    "fused_eager": {"graph": False},
    "four": {"four": True},
    "publish": {"q4_publish": True},
    "publish_four": {"q4_publish": True, "four": True},
    "global_merge": {"cluster_attn": False},
    "headproj": {"attn_oproj": True},
    "headproj3": {"attn_oproj": True, "four": True},
    "three": {"three": True},
    "unfused": {"unfused": True},
    "persistent": {"persistent": True},
}


@pytest.mark.parametrize("name", sorted(SMALL))
@pytest.mark.parametrize("mode", sorted(MODES))
def test_q4_layers_match_oracle(name, mode):
    w = SMALL[name]
    max_ctx = w.prefill + w.steps + 2
    d, host = workload.make_decoder(w, max_ctx=max_ctx, keep_host=True, **MODES[mode])
    xs = workload.step_inputs(w, w.steps)
    got = run_gpu(d, w, xs)
    d.close()
    ref = run_oracle(oracle_stack(w, host, max_ctx), w, xs)
    for s in range(w.steps):
        for l in range(w.n_layers):
            assert_close(got[s, l], ref[s, l], f"{name} {mode} step {s} layer {l}")


@pytest.mark.parametrize("mode", ["fused_graph", "publish", "headproj", "persistent"])
@pytest.mark.parametrize("kernel", [0, 2, 3, 4])
def test_q4_integer_block_dots_bit_exact(kernel, mode):
    w = SMALL["q4_gqa4_d64"]
    layer = 1
    max_ctx = w.prefill + 3
    d, host = workload.make_decoder(w, max_ctx=max_ctx, keep_host=True, **MODES[mode])
    km = max(w.hidden, w.ffn, w.n_q_heads * w.head_dim)
    qact = torch.zeros(w.n_layers, 4, km, dtype=torch.int8, device="cuda")
    qsc = torch.zeros(w.n_layers, 4, km // 32, dtype=torch.float32, device="cuda")
    K = {0: w.hidden, 2: w.n_q_heads * w.head_dim, 3: w.hidden, 4: w.ffn}[kernel]
    rows = tiled_rows_to_abi(w, kernel)
    dots = torch.full((len(rows), K // 32), -2**31, dtype=torch.int32, device="cuda")
    d.set_tap(None, qact, qsc)
    d.set_dot_tap(layer, kernel, dots)
    emb = torch.from_numpy(synth.step_input(w, 0)).cuda()
    out = torch.empty_like(emb)
    d.step(emb, w.prefill, out)
    d.sync_status()
    d.close()
    slot = {0: 0, 2: 1, 3: 2, 4: 3}[kernel]
    qx = qact[layer, slot, :K].cpu().numpy()
    gpu = dots.cpu().numpy().astype(np.int64)
    lw = host["layers"][layer]
    by_tensor = {}
    for t in {t for t, _ in rows}:
        packed, _ = lw.q4[t]
        by_tensor[t] = orc.q4_blockdots(packed, qx)       # int64, every ABI row
    ref = np.stack([by_tensor[t][r] for t, r in rows])
    assert np.array_equal(gpu, ref), f"{np.count_nonzero(gpu != ref)} block dots differ"


@pytest.mark.parametrize("mode", ["fused_graph", "four", "publish", "publish_four", "headproj"])
def test_q4_int8_activations_match_oracle_quantisation(mode):
    """Teacher-forced, slot by slot: the GPU's int8 codes against the oracle's
    own quantizer given the same layer input and the same upstream codes; every
    difference is a one-code flip of a value next to a rounding boundary."""
    w = SMALL["q4_mha_d128"]
    max_ctx = w.prefill + 3
    d, host = workload.make_decoder(w, max_ctx=max_ctx, keep_host=True, **MODES[mode])
    km = max(w.hidden, w.ffn, w.n_q_heads * w.head_dim)
    qact = torch.zeros(w.n_layers, 4, km, dtype=torch.int8, device="cuda")
    qsc = torch.zeros(w.n_layers, 4, km // 32, dtype=torch.float32, device="cuda")
    tap = torch.zeros(w.n_layers, w.hidden, device="cuda")
    d.set_tap(tap, qact, qsc)
    x = synth.step_input(w, 0)
    emb = torch.from_numpy(x).cuda()
    out = torch.empty_like(emb)
    d.step(emb, w.prefill, out)
    d.sync_status()
    rows = [d.read_kv(l, w.prefill, 1) for l in range(w.n_layers)]
    d.close()
    st = oracle_stack(w, host, max_ctx)
    inputs = [x.astype(np.float64)] + [tap[l].cpu().numpy().astype(np.float64)
                                       for l in range(w.n_layers - 1)]
    qa, qs = qact.cpu().numpy(), qsc.cpu().numpy()
    for l in range(w.n_layers):
        res = q4_code_flips(st, w, l, inputs[l], w.prefill, qa[l], qs[l], rows[l][0][:, 0],
                            rows[l][1][:, 0])
        for slot, (n, dist, K) in enumerate(res["slots"]):
            assert n <= max(1, Q4_FLIP_FRACTION[slot] * K), (l, Q4_SLOTS[slot], n)
            assert dist <= Q4_FLIP_DISTANCE, (l, Q4_SLOTS[slot], dist)
        n, dist, size = res["kv"]
        assert n <= 2e-3 * size and dist <= 1.0, (l, "KV row", n, dist)
