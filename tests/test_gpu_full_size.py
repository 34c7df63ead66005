"""Parity at the full workload sizes, in the launch configuration the benchmark
times (fused plan, CUDA graph, PDL, L2 look-ahead, cluster attention), against
the fp64 oracle on the same seeded weights, KV prefill and inputs.

- bf16 stacks (7B shape, 9B shape): every layer's output at every one of the
  benchmark's 128 decode steps against the free-running oracle, and the
  benchmark's own configuration (no taps) equal bit for bit to the tapped run;
- the int4/int8 stack, where floating point decides integers (the int8 codes
  of every GEMV input), checked in three parts:
  1. the integer decisions: slot by slot, the GPU's codes against the oracle's
     own quantizer given the same upstream codes; every difference must be a
     one-code flip of a value next to a rounding boundary;
  2. the float arithmetic around them: the free-running oracle taking the
     kernel's codes, every layer and step within the float tolerance (the
     dequantised outputs of the bit-exact integer dots);
  3. teacher-forced with its own codes and KV: every layer within the rel-L2
     bound, and within the max|err| bound wherever both sides decided the same
     codes; the free-running max|err| bound is a visible expected failure
     (a single flipped code moves elements of a hidden state that grows to
     |x| ~ 3e3 by more than 2e-2);
- int4: the integer block dots of one layer's four projections, bit-exact.

The oracle computes a token of these stacks in well under a second on the host
cores, so every layer of every step checked here is compared in full."""
import numpy as np
import pytest

from harness import (MAX_ABS, REL_L2, Q4_SLOTS, assert_close, errors, kv_row_flips, oracle_stack,
                     q4_code_flips, q4_slot_ks, run_gpu, run_oracle, tiled_rows_to_abi)
from oracle import oracle as orc
from transformer_layer_decode_gb300 import synth, workload

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

BENCH_STEPS = 128  # the benchmark's timed steps; KV capacity prefill + steps + 2
Q4_STEPS = 3
# Integer decisions of the int4 path: flips per slot and layer, as a fraction of
# the slot's codes, and the largest distance of a flipped value's quotient from
# the half-integer, in code units.  Measured at full width over 3 steps x 32
# layers: n1 <= 1, n2 <= 1, a <= 1 flips a layer; o <= 10 of 4096 (o is a
# softmax-weighted sum over ~2050 cached rows in fp32, so its rounding error
# relative to its block's absmax is the largest of the four).
Q4_FLIP_FRACTION = (1e-3, 5e-3, 1e-3, 1e-3)
Q4_FLIP_DISTANCE = 0.05
# The KV append's bf16 storage rounding: differing elements per row as a
# fraction of its elements; each must be a correct rounding of a value within
# 1e-5 x the head's RMS of the oracle's (excess <= 1, see bf16_flips).
KV_FLIP_FRACTION = 2e-3
KV_FLIP_DISTANCE = 1.0
KV_CHECK_STEPS = (0, BENCH_STEPS // 2, BENCH_STEPS - 1)


def _run_gpu_q4(d, w, xs):
    """Per-layer outputs [steps][layers][H] and each layer's int8 GEMV-input codes."""
    L, H = w.n_layers, w.hidden
    km = max(w.hidden, w.ffn, w.n_q_heads * w.head_dim)
    tap = torch.zeros(L, H, dtype=torch.float32, device="cuda")
    qact = torch.zeros(L, 4, km, dtype=torch.int8, device="cuda")
    qsc = torch.zeros(L, 4, km // 32, dtype=torch.float32, device="cuda")
    d.set_tap(tap, qact, qsc)
    emb = torch.empty(H, device="cuda")
    out = torch.empty(H, device="cuda")
    outs, codes = [], []
    for s, x in enumerate(xs):
        emb.copy_(torch.from_numpy(x))
        d.step(emb, w.prefill + s, out)
        d.sync_status()
        outs.append(tap.cpu().numpy())
        codes.append((qact.cpu().numpy(), qsc.cpu().numpy()))
    return np.stack(outs), codes


@pytest.mark.parametrize("name", ["stack32_h4096_mha", "stack40_h4096_gqa"])
def test_full_size_bf16_stack_every_benchmark_step(name):
    w = synth.WORKLOADS[name]
    max_ctx = w.prefill + BENCH_STEPS + 2
    d, host = workload.make_decoder(w, max_ctx=max_ctx, keep_host=True)
    xs = workload.step_inputs(w, BENCH_STEPS)
    final = run_gpu(d, w, xs, taps=False)  # exactly the benchmark's graph
    d.truncate_kv(w.prefill)
    got = run_gpu(d, w, xs)  # the same steps again with every layer tapped
    rows = [d.read_kv(l, w.prefill, BENCH_STEPS) for l in range(w.n_layers)]
    d.close()
    assert np.array_equal(got[:, -1], final), "taps changed the result"
    # the KV append: every appended row of the first, middle and last step,
    # against the oracle's storage rounding of k, v from the GPU's layer input
    st_kv = oracle_stack(w, host, max_ctx)
    worst_kv, n_kv = 0.0, 0
    for s in KV_CHECK_STEPS:
        for l in range(w.n_layers):
            inp = xs[s] if l == 0 else got[s, l - 1]
            n, dist, size = kv_row_flips(st_kv, l, inp, w.prefill + s, rows[l][0][:, s], rows[l][1][:, s])
            assert n <= KV_FLIP_FRACTION * size, f"step {s} layer {l}: {n} of {size} KV elements flipped"
            assert dist <= KV_FLIP_DISTANCE, f"step {s} layer {l}: a stored KV value off by {dist:.3e} x tolerance"
            worst_kv, n_kv = max(worst_kv, dist), n_kv + n
    print(f"{name}: KV append at steps {KV_CHECK_STEPS}: {n_kv} bf16 elements differ, largest "
          f"excess {worst_kv:.3e} x tolerance")
    ref = run_oracle(oracle_stack(w, host, max_ctx), w, xs)  # free-running
    worst = (0.0, 0.0, -1)
    for s in range(BENCH_STEPS):
        for l in range(w.n_layers):
            a, r = assert_close(got[s, l], ref[s, l], f"{name} step {s} layer {l}")
            if a > worst[0]:
                worst = (a, max(worst[1], r), s)
            worst = (worst[0], max(worst[1], r), worst[2])
    print(f"{name}: {BENCH_STEPS} steps x {w.n_layers} layers, worst max|err| {worst[0]:.3e} "
          f"(step {worst[2]}), worst rel-L2 {worst[1]:.3e}")


@pytest.fixture(scope="module")
def q4_run():
    w = synth.WORKLOADS["stack32_h4096_q4"]
    max_ctx = w.prefill + BENCH_STEPS + 2
    d, host = workload.make_decoder(w, max_ctx=max_ctx, keep_host=True)
    xs = workload.step_inputs(w, Q4_STEPS)
    final = run_gpu(d, w, xs, taps=False)
    d.truncate_kv(w.prefill)
    got, codes = _run_gpu_q4(d, w, xs)
    rows = [d.read_kv(l, w.prefill, Q4_STEPS) for l in range(w.n_layers)]
    d.close()
    free = run_oracle(oracle_stack(w, host, max_ctx), w, xs)
    return w, host, max_ctx, xs, final, got, codes, free, rows


def test_full_size_q4_stack(q4_run):
    w, host, max_ctx, xs, final, got, codes, free, rows = q4_run
    assert np.array_equal(got[:, -1], final), "taps changed the result"
    for s in range(Q4_STEPS):
        a, r = errors(got[s, -1], free[s, -1])
        assert r <= REL_L2, f"step {s}: free-running rel-L2 {r:.3e}"
        print(f"int4 stack free-running, step {s}: output max|err| {a:.3e} rel-L2 {r:.3e}")
    Ks = q4_slot_ks(w)
    # 2. the kernel's integer decisions fed to the free-running oracle
    stB = oracle_stack(w, host, max_ctx)
    worst_b = (0.0, 0.0)
    for s, x in enumerate(xs):
        pos = w.prefill + s
        qa, qs = codes[s]
        cur = np.asarray(x, np.float64)
        for l in range(w.n_layers):
            given = [(qa[l, i, :K], qs[l, i, :K // 32]) for i, K in enumerate(Ks)]
            cur = stB.layer_step(l, cur, pos, qgiven=given)
            a, r = assert_close(got[s, l], cur, f"step {s} layer {l} (oracle on the kernel's codes)")
            worst_b = (max(worst_b[0], a), max(worst_b[1], r))
        stB.kv_len = pos + 1
    # 1. and 3.: teacher-forced on the GPU's layer inputs
    stC = oracle_stack(w, host, max_ctx)   # its own codes and KV
    stD = oracle_stack(w, host, max_ctx)   # slot by slot
    worst_c, worst_c_same = (0.0, 0.0), 0.0
    flips = np.zeros((Q4_STEPS, w.n_layers, 4), np.int64)
    dist, kv_dist, kv_flips = 0.0, 0.0, 0
    for s, x in enumerate(xs):
        pos = w.prefill + s
        qa, qs = codes[s]
        for l in range(w.n_layers):
            inp = np.asarray(x if l == 0 else got[s, l - 1], np.float64)
            outC, tapsC = stC.layer_step(l, inp, pos, qtap=True)
            a, r = errors(got[s, l], outC)
            assert r <= REL_L2, f"step {s} layer {l} teacher-forced: rel-L2 {r:.3e}"
            same = all(np.array_equal(qa[l, i, :K], tapsC[i][0]) for i, K in enumerate(Ks))
            if same:
                assert a <= MAX_ABS, f"step {s} layer {l} teacher-forced, same codes: max|err| {a:.3e}"
                worst_c_same = max(worst_c_same, a)
            worst_c = (max(worst_c[0], a), max(worst_c[1], r))
            res = q4_code_flips(stD, w, l, inp, pos, qa[l], qs[l], rows[l][0][:, s], rows[l][1][:, s])
            for i, (n, dd, K) in enumerate(res["slots"]):
                flips[s, l, i] = n
                dist = max(dist, dd)
                assert n <= Q4_FLIP_FRACTION[i] * K, \
                    f"step {s} layer {l} {Q4_SLOTS[i]}: {n} of {K} codes flipped"
            n, dd, size = res["kv"]
            assert n <= KV_FLIP_FRACTION * size, f"step {s} layer {l}: {n} of {size} KV elements flipped"
            kv_dist, kv_flips = max(kv_dist, dd), kv_flips + n
        stC.kv_len = pos + 1
        stD.kv_len = pos + 1
    print(f"int4 stack, {Q4_STEPS} steps: oracle on the kernel's codes worst max|err| "
          f"{worst_b[0]:.3e} rel-L2 {worst_b[1]:.3e}; teacher-forced own codes worst max|err| "
          f"{worst_c[0]:.3e} (layers with the same codes {worst_c_same:.3e}) rel-L2 {worst_c[1]:.3e}")
    for i in range(4):
        f = flips[:, :, i]
        print(f"  {Q4_SLOTS[i]}: flips per layer max {f.max()} of {Ks[i]} "
              f"({f.max() / Ks[i]:.2e}), total {f.sum()} over {f.size} layer-steps")
    print(f"  largest distance of a flipped quotient from the half-integer: {dist:.3e}")
    print(f"  KV append: {kv_flips} bf16 elements differ, largest excess {kv_dist:.3e} x tolerance")
    assert dist <= Q4_FLIP_DISTANCE, f"a flipped code sits {dist:.3e} from its rounding boundary"
    assert kv_dist <= KV_FLIP_DISTANCE, f"a stored KV value off by {kv_dist:.3e} x tolerance"


@pytest.mark.xfail(reason="one flipped int8 code, decided on fp32 values by the kernel and fp64 "
                          "values by the oracle, moves single elements of a hidden state that "
                          "grows to |x| ~ 3e3 by more than 2e-2 once the stacks run free",
                   strict=False)
def test_full_size_q4_free_running_max_abs(q4_run):
    w, host, max_ctx, xs, final, got, codes, free, rows = q4_run
    for s in range(Q4_STEPS):
        for l in range(w.n_layers):
            assert_close(got[s, l], free[s, l], f"step {s} layer {l} free-running")


def test_full_size_q4_block_dots_bit_exact():
    w = synth.WORKLOADS["stack32_h4096_q4"].small(n_layers=2, name="q4_full_width_2layers")
    layer = 1
    max_ctx = w.prefill + BENCH_STEPS + 2
    d, host = workload.make_decoder(w, max_ctx=max_ctx, keep_host=True)
    km = max(w.hidden, w.ffn, w.n_q_heads * w.head_dim)
    qact = torch.zeros(w.n_layers, 4, km, dtype=torch.int8, device="cuda")
    qsc = torch.zeros(w.n_layers, 4, km // 32, dtype=torch.float32, device="cuda")
    d.set_tap(None, qact, qsc)
    lw = host["layers"][layer]
    for kernel, slot, K, tensors in ((0, 0, w.hidden, (synth.T_WQ, synth.T_WK, synth.T_WV)),
                                     (2, 1, w.n_q_heads * w.head_dim, (synth.T_WO,)),
                                     (3, 2, w.hidden, (synth.T_WGATE, synth.T_WUP)),
                                     (4, 3, w.ffn, (synth.T_WDOWN,))):
        n_rows = sum(lw.q4[t][0].shape[0] for t in tensors)
        dots = torch.full((n_rows, K // 32), -2**31, dtype=torch.int32, device="cuda")
        d.set_dot_tap(layer, kernel, dots)
        emb = torch.from_numpy(synth.step_input(w, 0)).cuda()
        out = torch.empty_like(emb)
        d.truncate_kv(w.prefill)
        d.step(emb, w.prefill, out)
        d.sync_status()
        qx = qact[layer, slot, :K].cpu().numpy()
        gpu = dots.cpu().numpy().astype(np.int64)
        rows = tiled_rows_to_abi(w, kernel)  # the dot tap is in the tiled row order
        by_tensor = {t: orc.q4_blockdots(lw.q4[t][0], qx) for t in tensors}
        ref = np.stack([by_tensor[t][r] for t, r in rows])
        assert np.array_equal(gpu, ref), f"kernel {kernel}: {np.count_nonzero(gpu != ref)} dots differ"
    d.close()
