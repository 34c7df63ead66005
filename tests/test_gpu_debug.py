"""Memory-safety checks that need no sanitizer (none can run here), on small
shapes of every plan:

- the debug build of the library (index checks compiled into the kernels:
  tiled offsets, stage sizes, attention chunks, KV rows, epilogue rows, split
  records; a failed check skips the access and raises the error flag with its
  source line);
- guard bands around every device buffer, buffers poisoned with NaN until
  written (a read of an unwritten byte reaches the results), KV rows past the
  KV length kept poisoned (an append outside its row is caught);

and the results still match the oracle."""
import numpy as np
import pytest

from harness import assert_close, oracle_stack, run_gpu, run_oracle
from transformer_layer_decode_gb300 import build as tld_build
from transformer_layer_decode_gb300 import dec, synth, workload

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

SHAPES = {
    "mha_d128": synth.Workload("mha_d128", 2, 512, 4, 4, 128, 1408, prefill=45, steps=3),
    "g8_d64_ragged": synth.Workload("g8_d64_ragged", 2, 264, 16, 2, 64, 1000, prefill=200, steps=3),
    "q4_gqa4": synth.Workload("q4_gqa4", 2, 512, 8, 2, 64, 1408, prefill=100, steps=2, weight_fmt="q4"),
}
PLANS = {
    "fused": {},
    "global_merge": {"cluster_attn": False},
    "three": {"three": True},
    "persistent": {"persistent": True},
    "unfused": {"unfused": True},
    "paged": {"paged_kv": True},
    "q4_publish": {"q4_publish": True},  # int4 shapes: inputs published by their producers
    "headproj": {"attn_oproj": True},
    "headproj3": {"attn_oproj": True, "four": True},
}


@pytest.fixture(scope="module")
def debug_lib():
    return tld_build.build(debug=True)


@pytest.mark.parametrize("plan", sorted(PLANS))
@pytest.mark.parametrize("name", sorted(SHAPES))
def test_debug_build_with_guards(debug_lib, name, plan):
    w = SHAPES[name]
    max_ctx = w.prefill + w.steps + 3
    d = dec.Decoder(workload.shape_of(w, max_ctx), guards=True, lib_path=debug_lib, **PLANS[plan])
    if plan == "paged":
        d.set_page_table(np.random.default_rng(3).permutation(d.info().n_pages))
    host = {"layers": [], "kv": []}
    for l in range(w.n_layers):
        lw = synth.layer_weights(w, l)
        workload.load_layer(d, w, l, lw)
        k, v = synth.kv_bf16(w, l, w.prefill)
        d.load_kv(l, k, v, w.prefill)
        host["layers"].append(lw)
        host["kv"].append((k, v))
    d.check_guards()                         # loading wrote only inside its buffers
    xs = workload.step_inputs(w, w.steps)
    got = run_gpu(d, w, xs)                  # every step: sync_status (index checks, waits)
    d.check_guards()                         # guards intact, rows past the KV length untouched
    d.truncate_kv(w.prefill)                 # rows past the prefill poisoned again
    d.check_guards()
    again = run_gpu(d, w, xs)
    d.check_guards()
    d.close()
    assert np.array_equal(got, again)
    ref = run_oracle(oracle_stack(w, host, max_ctx), w, xs)
    for s in range(w.steps):
        for l in range(w.n_layers):
            assert_close(got[s, l], ref[s, l], f"{name} {plan} step {s} layer {l}")


def test_guard_check_needs_guards():
    w = SHAPES["mha_d128"]
    d = dec.Decoder(workload.shape_of(w, 64))
    with pytest.raises(dec.DecError) as e:
        d.check_guards()
    assert e.value.code == dec.DEC_ERR_STATE
    d.close()
