"""dec_attention_noalloc against the decoder's own attention, through the C ABI.

Some callers cannot call cudaMalloc (their device memory belongs to another
allocator, or they run under a no-allocation rule after start-up), so the
library offers the decode attention kernel with its scratch in a fixed device
array.  This test checks that entry point's output against the attention that
dec_step computes, on two calls in a row.

The decoder's attention output is made observable through dec_step: one layer
with Wq = I, Wk = Wv = 0, Wo = I, Wdown = 0 and unit norm weights gives
out = x + attention(RoPE(rmsnorm(x))), with zero k/v appended at each step.
"""
import numpy as np
import pytest

from harness import assert_close
from transformer_layer_decode_gb300 import dec

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

H, NQ, NKV, D, F = 256, 4, 2, 64, 64
PREFILL = 300           # several 128-row chunks per head: heads split over CTAs
MAX_CTX = PREFILL + 4
EPS, THETA = 1e-6, 1e4
ONE = 0x3F80            # bf16 1.0


def _bf16(a: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16).view(
        torch.int16).numpy().view(np.uint16)


def _rope(h: np.ndarray, pos: int) -> np.ndarray:
    """Rotate-half RoPE of [heads][D] in double."""
    half = D // 2
    ang = pos * THETA ** (-2.0 * np.arange(half) / D)
    c, s = np.cos(ang), np.sin(ang)
    a, b = h[:, :half], h[:, half:]
    return np.concatenate([a * c - b * s, a * s + b * c], axis=1)


def test_noalloc_attention_matches_decoder_attention():
    rng = np.random.default_rng(7)
    d = dec.Decoder(dec.Shape(1, H, NQ, NKV, D, F, MAX_CTX, EPS, THETA))
    eye = np.where(np.eye(H, dtype=bool), ONE, 0).astype(np.uint16)
    d.load_weights(0, dec.DEC_T_ATTN_NORM, np.full(H, ONE, np.uint16))
    d.load_weights(0, dec.DEC_T_FFN_NORM, np.full(H, ONE, np.uint16))
    d.load_weights(0, dec.DEC_T_WQ, eye)
    d.load_weights(0, dec.DEC_T_WK, np.zeros((NKV * D, H), np.uint16))
    d.load_weights(0, dec.DEC_T_WV, np.zeros((NKV * D, H), np.uint16))
    d.load_weights(0, dec.DEC_T_WO, eye)
    d.load_weights(0, dec.DEC_T_WGATE, _bf16(rng.normal(0, 0.02, (F, H))))
    d.load_weights(0, dec.DEC_T_WUP, _bf16(rng.normal(0, 0.02, (F, H))))
    d.load_weights(0, dec.DEC_T_WDOWN, np.zeros((H, F), np.uint16))
    kp = _bf16(rng.normal(0, 1, (NKV, PREFILL, D)))
    vp = _bf16(rng.normal(0, 1, (NKV, PREFILL, D)))
    d.load_kv(0, kp, vp)

    # the same cache for the no-alloc call: prefill rows, then zero rows appended
    kc = np.zeros((NKV, MAX_CTX, D), np.uint16)
    vc = np.zeros((NKV, MAX_CTX, D), np.uint16)
    kc[:, :PREFILL], vc[:, :PREFILL] = kp, vp
    kc_dev = torch.from_numpy(kc.view(np.int16)).cuda()
    vc_dev = torch.from_numpy(vc.view(np.int16)).cuda()

    emb = torch.empty(H, device="cuda")
    out = torch.empty(H, device="cuda")
    o_dev = torch.empty(NQ * D, device="cuda")
    for call in range(2):                         # two calls in a row
        pos = PREFILL + call
        x = rng.normal(0, 1, H).astype(np.float32)
        emb.copy_(torch.from_numpy(x))
        d.step(emb, pos, out)
        d.sync_status()
        o_decoder = out.cpu().numpy().astype(np.float64) - x    # out = x + attention

        n1 = x.astype(np.float64) / np.sqrt(np.mean(x.astype(np.float64) ** 2) + EPS)
        q = torch.from_numpy(_rope(n1.reshape(NQ, D), pos).astype(np.float32).ravel()).cuda()
        o_dev.fill_(float("nan"))
        dec.attention_noalloc(q, kc_dev, vc_dev, NQ, NKV, D, MAX_CTX, pos + 1, o_dev)
        torch.cuda.synchronize()
        got = o_dev.cpu().numpy()
        assert np.all(np.isfinite(got))
        assert_close(got, o_decoder, f"no-alloc attention, call {call + 1}")
    d.close()


def test_noalloc_rejects_sizes_beyond_its_limits():
    q = torch.zeros(8 * 64, device="cuda")
    kv = torch.zeros(100 * 8 * 64, dtype=torch.int16, device="cuda")
    o = torch.empty_like(q)
    with pytest.raises(dec.DecError) as e:
        dec.attention_noalloc(q, kv, kv, 8, 1, 96, 100, 10, o)      # head_dim 96
    assert e.value.code == dec.DEC_ERR_SHAPE
    with pytest.raises(dec.DecError) as e:
        dec.attention_noalloc(q, kv, kv, 8, 1, 64, 100, 101, o)     # n > ctx_stride
    assert e.value.code == dec.DEC_ERR_ARG
    with pytest.raises(dec.DecError) as e:
        dec.attention_noalloc(q, kv, kv, 8, 128, 64, 100, 10, o)    # > 64 KV heads
    assert e.value.code == dec.DEC_ERR_SHAPE
