"""GPU parity: the CUDA path through the C ABI against the fp64 oracle on the
same seeded inputs, per layer and per step (max|err| <= 2e-2, rel-L2 <= 5e-3),
plus plan equivalence, determinism and graph / eager agreement."""
import numpy as np
import pytest

from harness import assert_close, oracle_stack, run_gpu, run_oracle
from transformer_layer_decode_gb300 import dec, synth, workload

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)


def _check(w, steps, *, max_ctx=None, **plan):
    max_ctx = max_ctx or w.prefill + steps + 2
    d, host = workload.make_decoder(w, max_ctx=max_ctx, keep_host=True, **plan)
    xs = workload.step_inputs(w, steps)
    got = run_gpu(d, w, xs)
    d.close()
    ref = run_oracle(oracle_stack(w, host, max_ctx), w, xs)
    worst = (0.0, 0.0)
    for s in range(steps):
        for l in range(w.n_layers):
            a, r = assert_close(got[s, l], ref[s, l], f"{w.name} step {s} layer {l}")
            worst = (max(worst[0], a), max(worst[1], r))
    return got, worst


def test_layer_h512_single_step():
    """One layer, hidden 512, GQA 8/2, d 64, F 1408, decode at pos 127."""
    _check(synth.WORKLOADS["layer_h512"], 1)


SMALL = {
    # ragged K tiles (264 = 256 + 8; 1000 = 3*256 + 232), GQA 2, empty prefill (KV length 1)
    "ragged_g2_empty": synth.Workload("ragged_g2_empty", 2, 264, 4, 2, 64, 1000, prefill=0, steps=3),
    # MHA, head_dim 128, prefill not a multiple of the chunk
    "mha_d128": synth.Workload("mha_d128", 2, 512, 4, 4, 128, 1408, prefill=45, steps=3),
    # GQA 8, fewer rows than SMs
    "g8_d64": synth.Workload("g8_d64", 1, 256, 16, 2, 64, 512, prefill=200, steps=2),
    # GQA 4, d 128, context spanning many chunks and CTAs
    "g4_d128_long": synth.Workload("g4_d128_long", 1, 1024, 8, 2, 128, 2816, prefill=1500, steps=2),
}


MODES = {
    "fused_graph": {},                                   # five kernels, cluster attention
    "fused_eager": {"graph": False},
    "global_merge": {"cluster_attn": False},
    "four": {"four": True},                              # four kernels per layer
    "three": {"three": True},                            # three kernels per layer
    "three_eager": {"three": True, "graph": False},
    "unfused": {"unfused": True},
    "persistent": {"persistent": True},
    # attention + o-projection by KV-head group in one cluster launch
    "headproj": {"attn_oproj": True},
    "headproj_eager": {"attn_oproj": True, "graph": False},
    "headproj3": {"attn_oproj": True, "four": True},
}


@pytest.mark.parametrize("name", sorted(SMALL))
@pytest.mark.parametrize("mode", sorted(MODES))
def test_small_shapes(name, mode):
    _check(SMALL[name], SMALL[name].steps, **MODES[mode])


INTERLEAVED = {
    "inter_g4_d128": synth.Workload("inter_g4_d128", 2, 512, 8, 2, 128, 1408, prefill=70, steps=3,
                                    rope_interleaved=True),
    "inter_q4_mha_d64": synth.Workload("inter_q4_mha_d64", 2, 512, 8, 8, 64, 1408, prefill=30,
                                       steps=2, weight_fmt="q4", rope_interleaved=True),
}


@pytest.mark.parametrize("name", sorted(INTERLEAVED))
@pytest.mark.parametrize("mode", ["fused_graph", "headproj", "three", "unfused", "persistent"])
def test_rope_interleaved_pairs(name, mode):
    """RoPE on pairs (2i, 2i+1): every plan against the oracle's interleaved chain."""
    w = INTERLEAVED[name]
    _check(w, w.steps, **MODES[mode])


@pytest.mark.parametrize("mode", ["fused_graph", "headproj", "four", "three", "persistent"])
def test_stack16_h2048_all_steps(mode):
    """16-layer 1B-shape stack, 64 steps from pos 1023, every layer at every step."""
    w = synth.WORKLOADS["stack16_h2048"]
    _, worst = _check(w, w.steps, **MODES[mode])
    print("stack16 (%s) worst max|err| %.3e rel-L2 %.3e" % ((mode,) + worst))


def test_plans_agree_and_are_deterministic():
    w = SMALL["mha_d128"]
    xs = workload.step_inputs(w, 3)
    outs = {}
    for key, kw in {"graph": {}, "graph2": {}, "eager": {"graph": False},
                    "no_l2_ahead": {"l2_ahead": False}, "no_pdl": {"pdl": False},
                    "global_merge": {"cluster_attn": False},
                    "three": {"three": True}, "three_eager": {"three": True, "graph": False},
                    "four": {"four": True},
                    "headproj": {"attn_oproj": True},
                    "headproj_eager": {"attn_oproj": True, "graph": False},
                    "headproj_no_pdl": {"attn_oproj": True, "pdl": False},
                    "headproj3": {"attn_oproj": True, "four": True},
                    "persistent": {"persistent": True},
                    "persistent_eager": {"persistent": True, "graph": False},
                    "unfused": {"unfused": True}}.items():
        d, _ = workload.make_decoder(w, max_ctx=64, **kw)
        outs[key] = run_gpu(d, w, xs)
        d.close()
    assert np.array_equal(outs["graph"], outs["graph2"]), "fused plan not run-to-run identical"
    assert np.array_equal(outs["graph"], outs["eager"]), "graph replay differs from eager launch"
    assert np.array_equal(outs["graph"], outs["no_l2_ahead"]), "the L2 look-ahead changed results"
    assert np.array_equal(outs["graph"], outs["no_pdl"]), "dependent launch changed results"
    assert np.array_equal(outs["three"], outs["three_eager"])
    # gate/up + down in one launch: the same split and arithmetic as two launches
    assert np.array_equal(outs["graph"], outs["four"]), "four vs five kernels differ"
    # the three-kernel plan and the persistent plan run the same split and the
    # same per-phase arithmetic (attention with the GEMV kernels' warp count)
    assert np.array_equal(outs["three"], outs["persistent"]), "persistent differs from three"
    assert np.array_equal(outs["persistent"], outs["persistent_eager"])
    # attention + o-projection in one launch: deterministic group order
    assert np.array_equal(outs["headproj"], outs["headproj_eager"])
    assert np.array_equal(outs["headproj"], outs["headproj_no_pdl"])
    assert np.array_equal(outs["headproj"], outs["headproj3"]), "two-phase FFN changed results"
    for s in range(3):
        for l in range(w.n_layers):
            assert_close(outs["graph"][s, l], outs["headproj"][s, l], f"five vs headproj {s},{l}")
    for s in range(3):
        for l in range(w.n_layers):
            assert_close(outs["graph"][s, l], outs["three"][s, l], f"five vs three {s},{l}")
            assert_close(outs["graph"][s, l], outs["global_merge"][s, l], f"cluster vs global {s},{l}")
    for s in range(3):
        for l in range(w.n_layers):
            assert_close(outs["graph"][s, l], outs["unfused"][s, l], f"fused vs unfused {s},{l}")


def test_residual_wiring_zero_projections():
    """Wo = 0 and Wd = 0: every layer returns its input exactly."""
    w = SMALL["mha_d128"]
    d = dec.Decoder(workload.shape_of(w, 64))
    for l in range(w.n_layers):
        lw = synth.layer_weights(w, l)
        lw.mats[synth.T_WO][:] = 0
        lw.mats[synth.T_WDOWN][:] = 0
        workload.load_layer(d, w, l, lw)
        k, v = synth.kv_bf16(w, l, w.prefill)
        d.load_kv(l, k, v)
    xs = workload.step_inputs(w, 2)
    got = run_gpu(d, w, xs)
    d.close()
    for s in range(2):
        for l in range(w.n_layers):
            assert np.array_equal(got[s, l], xs[s])


@pytest.mark.parametrize("mode", ["fused_graph", "headproj", "headproj3", "three", "persistent"])
def test_io_pointers_can_change_between_steps(mode):
    """The captured graph is re-pointed when the caller passes new buffers."""
    w = SMALL["ragged_g2_empty"]
    xs = workload.step_inputs(w, 3)
    d_ref, _ = workload.make_decoder(w, max_ctx=16, **{**MODES[mode], "graph": False})
    ref = run_gpu(d_ref, w, xs, taps=False)
    d_ref.close()
    d, _ = workload.make_decoder(w, max_ctx=16, **MODES[mode])
    outs = []
    for s in range(3):
        emb = torch.from_numpy(xs[s]).cuda()          # a fresh buffer every step
        out = torch.full((w.hidden,), float("nan"), device="cuda")
        d.step(emb, s, out)
        d.sync_status()
        outs.append(out.cpu().numpy())
    d.close()
    assert np.array_equal(np.stack(outs), ref)


def test_step_errors_on_gpu():
    w = SMALL["ragged_g2_empty"]
    d, _ = workload.make_decoder(w, max_ctx=4)
    emb = torch.zeros(w.hidden, device="cuda")
    out = torch.zeros(w.hidden, device="cuda")
    with pytest.raises(dec.DecError) as e:
        d.step(emb, 1, out)                      # pos != KV length
    assert e.value.code == dec.DEC_ERR_POS
    for p in range(4):
        d.step(emb, p, out)
    with pytest.raises(dec.DecError) as e:
        d.step(emb, 4, out)                      # cache full
    assert e.value.code == dec.DEC_ERR_CTX
    d.truncate_kv(1)
    d.step(emb, 1, out)
    d.sync_status()
    with pytest.raises(dec.DecError) as e:
        d.load_weights(0, dec.DEC_T_WQ, np.zeros(7, np.uint16))   # wrong size
    assert e.value.code == dec.DEC_ERR_ARG
    d.close()
    fresh = dec.Decoder(workload.shape_of(w, 4))
    with pytest.raises(dec.DecError) as e:
        fresh.step(emb, 0, out)                  # weights missing
    assert e.value.code == dec.DEC_ERR_STATE
    fresh.close()


PAGED = {
    "paged_g4_d128": synth.Workload("paged_g4_d128", 2, 512, 8, 2, 128, 1408, prefill=150, steps=3),
    "paged_mha_d64": synth.Workload("paged_mha_d64", 2, 512, 8, 8, 64, 1408, prefill=300, steps=3),
    "paged_q4_g2_d64": synth.Workload("paged_q4_g2_d64", 1, 512, 4, 2, 64, 1408, prefill=200,
                                      steps=2, weight_fmt="q4"),
}


@pytest.mark.parametrize("name", sorted(PAGED))
@pytest.mark.parametrize("mode", ["fused_graph", "global_merge", "headproj", "four", "three",
                                  "persistent"])
def test_paged_kv_matches_contiguous_and_oracle(name, mode):
    """Kernel to parts: the fused QKV kernel writing the rotated k and the v of
    each token into its KV page (a shuffled page table), and attention reading
    the pages, give bit for bit what the same plan gives on the contiguous cache,
    and the oracle's result; the appended rows read back equal; rows move with
    their pages when the table changes between steps."""
    w = PAGED[name]
    max_ctx = w.prefill + w.steps + 40
    xs = workload.step_inputs(w, w.steps)
    d, host = workload.make_decoder(w, max_ctx=max_ctx, keep_host=True, **MODES[mode])
    flat = run_gpu(d, w, xs)
    flat_rows = [d.read_kv(l, 0, w.prefill + w.steps) for l in range(w.n_layers)]
    d.close()
    d, _ = workload.make_decoder(w, max_ctx=max_ctx, paged_kv=True, **MODES[mode])
    n_pages = d.info().n_pages
    rng = np.random.default_rng(5)
    d.set_page_table(rng.permutation(n_pages))
    half = w.steps // 2
    got = [run_gpu(d, w, xs[:half])] if half else []
    d.set_page_table(rng.permutation(n_pages))  # cached rows move with their pages
    emb = torch.empty(w.hidden, device="cuda")
    out = torch.empty(w.hidden, device="cuda")
    tap = torch.zeros(w.n_layers, w.hidden, device="cuda")
    d.set_tap(tap)
    rest = []
    for s in range(half, w.steps):
        emb.copy_(torch.from_numpy(xs[s]))
        d.step(emb, w.prefill + s, out)
        d.sync_status()
        rest.append(tap.cpu().numpy().copy())
    got = np.concatenate(got + [np.stack(rest)]) if got else np.stack(rest)
    paged_rows = [d.read_kv(l, 0, w.prefill + w.steps) for l in range(w.n_layers)]
    d.close()
    assert np.array_equal(got, flat), "paged and contiguous caches give different results"
    for l in range(w.n_layers):
        assert np.array_equal(paged_rows[l][0], flat_rows[l][0])
        assert np.array_equal(paged_rows[l][1], flat_rows[l][1])
    ref = run_oracle(oracle_stack(w, host, max_ctx), w, xs)
    for s in range(w.steps):
        for l in range(w.n_layers):
            assert_close(got[s, l], ref[s, l], f"{name} {mode} paged step {s} layer {l}")


def _rope_rows(h: np.ndarray, pos: int, d: int, theta: float) -> np.ndarray:
    """Rotate-half RoPE of [heads][d] in double."""
    half = d // 2
    ang = pos * theta ** (-2.0 * np.arange(half) / d)
    c, s = np.cos(ang), np.sin(ang)
    a, b = h[:, :half], h[:, half:]
    return np.concatenate([a * c - b * s, a * s + b * c], axis=1)


@pytest.mark.parametrize("hd,nq,nkv", [(128, 2, 2), (64, 4, 2)])
@pytest.mark.parametrize("mode", ["fused_graph", "headproj", "global_merge"])
def test_attention_rising_scores_through_the_step(hd, nq, nkv, mode):
    """The decoder's own attention (cluster kernels with records pushed or
    exchanged, and the flat grid) on a prefilled context whose scores for query
    head 0 climb by 20 per chunk over periods of 8 chunks: the online softmax's
    reference max moves past its slack of 8 at almost every chunk each CTA
    streams (~8 chunks a CTA), so the rescaling path keeps running.  One layer
    with Wq = Wo = I, Wk = Wv = Wdown = 0 and unit norms gives
    out = x + attention(RoPE(rmsnorm(x))); compared with the oracle's attention
    head by head."""
    from oracle import oracle as orc
    eps, theta, one = 1e-6, 1e4, 0x3F80
    H, F = nq * hd, 64
    ch = 16384 // (2 * hd)                 # rows of one 16 KB K chunk
    prefill = 128 * ch                     # 128 chunks a head: ~8 a CTA at 16 CTAs a head
    max_ctx = prefill + 4
    rng = np.random.default_rng(hd * 10 + nq)

    def bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16).view(
            torch.int16).numpy().view(np.uint16)

    x = rng.normal(0, 1, H).astype(np.float32)
    pos = prefill
    n1 = x.astype(np.float64) / np.sqrt(np.mean(x.astype(np.float64) ** 2) + eps)
    q = _rope_rows(n1.reshape(nq, hd), pos, hd, theta)
    scale = 1.0 / np.sqrt(hd)
    t = np.arange(prefill)
    target = 20.0 * (t % (8 * ch)) / ch
    g0 = orc.kv_head_of(0, nq, nkv)
    kp = np.empty((nkv, prefill, hd), np.float32)
    kp[g0] = (target / scale)[:, None] * (q[0] / (q[0] @ q[0]))[None, :]
    for g in range(nkv):
        if g != g0:
            kp[g] = rng.normal(0, 1, (prefill, hd))
    kp = bf16(kp)
    vp = bf16(rng.normal(0, 1, (nkv, prefill, hd)))
    k64 = torch.from_numpy(kp.view(np.int16)).view(torch.bfloat16).double().numpy()
    top = ((k64[g0] @ q[0]) * scale).reshape(-1, ch).max(axis=1)
    steps = np.diff(top)[(np.arange(len(top) - 1) + 1) % 8 != 0]
    assert steps.min() > 8.0               # the construction, on the stored keys

    d = dec.Decoder(dec.Shape(1, H, nq, nkv, hd, F, max_ctx, eps, theta), **MODES[mode])
    eye = np.where(np.eye(H, dtype=bool), one, 0).astype(np.uint16)
    d.load_weights(0, dec.DEC_T_ATTN_NORM, np.full(H, one, np.uint16))
    d.load_weights(0, dec.DEC_T_FFN_NORM, np.full(H, one, np.uint16))
    d.load_weights(0, dec.DEC_T_WQ, eye)
    d.load_weights(0, dec.DEC_T_WK, np.zeros((nkv * hd, H), np.uint16))
    d.load_weights(0, dec.DEC_T_WV, np.zeros((nkv * hd, H), np.uint16))
    d.load_weights(0, dec.DEC_T_WO, eye)
    d.load_weights(0, dec.DEC_T_WGATE, bf16(rng.normal(0, 0.02, (F, H))))
    d.load_weights(0, dec.DEC_T_WUP, bf16(rng.normal(0, 0.02, (F, H))))
    d.load_weights(0, dec.DEC_T_WDOWN, np.zeros((H, F), np.uint16))
    d.load_kv(0, kp, vp)
    emb = torch.from_numpy(x).cuda()
    out = torch.empty(H, device="cuda")
    d.step(emb, pos, out)
    d.sync_status()
    got = out.cpu().numpy().astype(np.float64) - x      # out = x + attention
    d.close()
    kz = np.concatenate([kp, np.zeros((nkv, 1, hd), np.uint16)], axis=1)   # the appended row: k = v = 0
    vz = np.concatenate([vp, np.zeros((nkv, 1, hd), np.uint16)], axis=1)
    for h in range(nq):
        g = orc.kv_head_of(h, nq, nkv)
        ref = orc.attention_head(q[h], kz[g], vz[g])
        assert_close(got[h * hd:(h + 1) * hd], ref, f"rising scores through the step, {mode}, hd {hd}, head {h}",
                     max_abs=1e-3, rel_l2=1e-4)
