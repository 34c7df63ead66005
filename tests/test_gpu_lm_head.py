"""The LM head and greedy token after the stack, through the C ABI, against the
oracle: the final RMSNorm, the vocabulary projection (32000 x 4096 after the
7B-shape stack) and the greedy choice, inside the captured token graph.

The token is an integer decided by floating point (an argmax): the oracle
decides it on its fp64 logits of the GPU's final hidden state; where the two
choices differ, the oracle's logits of both rows must be a near tie within the
fp32 arithmetic's error, and otherwise the choices must be equal."""
import numpy as np
import pytest

from harness import assert_close
from oracle import oracle as orc
from transformer_layer_decode_gb300 import synth, workload

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

VOCAB = 32000
TIE_TOL = 1e-4  # fp32 error of a 4096-term logit (|logit| ~ 1), with margin


def _decode_tokens(d, w, xs, nw, W):
    H = w.hidden
    tok = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    logits = torch.empty(W.shape[0], dtype=torch.float32, device="cuda")
    d.load_lm_head(nw, W)
    d.set_token_out(tok, logits)
    emb = torch.empty(H, device="cuda")
    out = torch.empty(H, device="cuda")
    res = []
    for s, x in enumerate(xs):
        emb.copy_(torch.from_numpy(x))
        d.step(emb, w.prefill + s, out)
        d.sync_status()
        res.append((int(tok.item()), logits.cpu().numpy().copy(), out.cpu().numpy().copy()))
    return res


def _check_against_oracle(res, nw, W, eps, what):
    for s, (tok, logits, hidden) in enumerate(res):
        tok_o, logits_o = orc.lm_head(hidden.astype(np.float64), nw, W, eps)
        assert_close(logits, logits_o, f"{what} step {s} logits", max_abs=1e-3, rel_l2=1e-5)
        if tok != tok_o:
            gap = abs(logits_o[tok] - logits_o[tok_o])
            assert gap <= TIE_TOL, f"{what} step {s}: token {tok} vs {tok_o}, logit gap {gap:.3e}"
            print(f"{what} step {s}: near tie {tok} / {tok_o} (gap {gap:.2e})")


def test_lm_head_after_the_7b_stack():
    w = synth.WORKLOADS["stack32_h4096_mha"]
    nw, W = synth.lm_head(w, VOCAB)
    xs = workload.step_inputs(w, 3)
    d, _ = workload.make_decoder(w, max_ctx=w.prefill + 8)
    graph = _decode_tokens(d, w, xs, nw, W)
    d.close()
    _check_against_oracle(graph, nw, W, w.rms_eps, "graph")
    d, _ = workload.make_decoder(w, max_ctx=w.prefill + 8, graph=False)
    eager = _decode_tokens(d, w, xs, nw, W)
    d.close()
    for (tg, lg, hg), (te, le, he) in zip(graph, eager):
        assert tg == te and np.array_equal(lg, le) and np.array_equal(hg, he)
    print("tokens:", [t for t, _, _ in graph])


@pytest.mark.parametrize("mode", ["fused", "three", "unfused", "persistent"])
def test_lm_head_every_plan_and_ties(mode):
    """A small stack; two identical LM head rows at the same position within
    their row blocks (so their fp32 logits are bit-identical) made the largest:
    the lower row wins."""
    w = synth.Workload("lm_small", 2, 512, 8, 2, 64, 1408, prefill=40, steps=3)
    kw = {"fused": {}, "three": {"three": True}, "unfused": {"unfused": True},
          "persistent": {"persistent": True}}[mode]
    nw, W = synth.lm_head(w, 4096)
    xs = workload.step_inputs(w, 3)
    d, _ = workload.make_decoder(w, max_ctx=w.prefill + 8, **kw)
    res = _decode_tokens(d, w, xs, nw, W)
    _check_against_oracle(res, nw, W, w.rms_eps, mode)
    # ties: rows 4*100+1 and 4*900+1 equal and largest for the last hidden state
    hidden = res[-1][2].astype(np.float64)
    _, logits_o = orc.lm_head(hidden, nw, W, w.rms_eps)
    top = int(np.argmax(logits_o))
    Wt = W.copy()
    big = (synth.bf16_to_f32(W[top]) * 4.0).astype(np.float32)
    row = torch.from_numpy(big).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    Wt[401] = row
    Wt[3601] = row
    d.truncate_kv(w.prefill)
    res_t = _decode_tokens(d, w, xs, nw, Wt)
    d.close()
    tok_t, logits_t, _ = res_t[-1]
    assert logits_t[401] == logits_t[3601]
    assert tok_t == 401, tok_t
