"""dec_attention_noalloc against the decoder's own attention and against the
fp64 oracle, through the C ABI.

Some callers cannot call cudaMalloc (their device memory belongs to another
allocator, or they run under a no-allocation rule after start-up), so the
library offers the decode attention kernel with its scratch in a fixed device
array.  These tests check that entry point's output against the attention that
dec_step computes and against the oracle's attention, on two calls in a row,
and that calls whose partial records would not fit the array are refused.

The decoder's attention output is made observable through dec_step: one layer
with Wq = I, Wk = Wv = 0, Wo = I, Wdown = 0 and unit norm weights gives
out = x + attention(RoPE(rmsnorm(x))), with zero k/v appended at each step.
"""
import numpy as np
import pytest

from harness import assert_close
from oracle import oracle as orc
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


@pytest.mark.parametrize("nq,nkv,hd,n", [(32, 4, 128, 777), (8, 4, 64, 300), (16, 16, 128, 129)])
def test_noalloc_attention_matches_oracle(nq, nkv, hd, n):
    """GQA 8 at head_dim 128, GQA 2 at 64 and MHA at 128 against the oracle's
    attention head by head, two calls in a row (the second one longer)."""
    rng = np.random.default_rng(nq * 1000 + hd)
    ctx = n + 8
    kc = _bf16(rng.normal(0, 1, (nkv, ctx, hd)))
    vc = _bf16(rng.normal(0, 1, (nkv, ctx, hd)))
    kc_dev = torch.from_numpy(kc.view(np.int16)).cuda()
    vc_dev = torch.from_numpy(vc.view(np.int16)).cuda()
    o_dev = torch.empty(nq * hd, device="cuda")
    for call, length in enumerate((n, n + 5)):
        q = rng.normal(0, 1, (nq, hd)).astype(np.float32)
        o_dev.fill_(float("nan"))
        dec.attention_noalloc(torch.from_numpy(q.ravel()).cuda(), kc_dev, vc_dev, nq, nkv, hd,
                              ctx, length, o_dev)
        dec.noalloc_sync_status()
        got = o_dev.cpu().numpy().reshape(nq, hd)
        for h in range(nq):
            g = orc.kv_head_of(h, nq, nkv)
            ref = orc.attention_head(q[h].astype(np.float64), kc[g, :length], vc[g, :length])
            assert_close(got[h], ref, f"no-alloc vs oracle, {nq}/{nkv} hd {hd}, call {call + 1} head {h}",
                         max_abs=1e-4, rel_l2=1e-5)


def test_noalloc_refuses_records_beyond_its_array():
    """64 q / 8 KV heads at head_dim 128: the split records of one call need
    grid * 2 * 8 * 132 floats, more than the 2^18 the array holds on a GPU with
    more than 124 SMs; the call is refused with DEC_ERR_SHAPE and queues nothing."""
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    grid = min(n_sm, 31 * 8)
    if grid * 2 * 8 * 132 <= 1 << 18:
        pytest.skip("this GPU's grid fits the records")
    q = torch.zeros(64 * 128, device="cuda")
    kv = torch.zeros(8 * 64 * 128, dtype=torch.int16, device="cuda")
    o = torch.full_like(q, 7.0)
    with pytest.raises(dec.DecError) as e:
        dec.attention_noalloc(q, kv, kv, 64, 8, 128, 64, 10, o)
    assert e.value.code == dec.DEC_ERR_SHAPE
    torch.cuda.synchronize()
    assert torch.all(o == 7.0)                 # nothing ran
    dec.noalloc_sync_status()


@pytest.mark.parametrize("hd,nq,nkv", [(128, 2, 2), (64, 4, 2)])
def test_noalloc_attention_rising_scores_against_oracle(hd, nq, nkv):
    """Scores that climb by 20 per attention chunk over a period of 8 chunks
    (far past the online softmax's slack of 8) move the running max at almost
    every chunk a CTA streams, so the rescaling path runs again and again (a
    CTA streams ~8 chunks of the 40 000-row context); the other KV head's keys
    are random (one rescale, at its first chunk).  Compared head by head with
    the oracle's attention."""
    rng = np.random.default_rng(hd + nq)
    n = 40000
    ctx = n + 8
    ch = 16384 // (2 * hd)  # rows of one 16 KB K chunk
    q = rng.normal(0, 1, (nq, hd)).astype(np.float32)
    scale = 1.0 / np.sqrt(hd)
    t = np.arange(ctx)
    target = 20.0 * (t % (8 * ch)) / ch  # scores wanted for query head 0
    kc = np.empty((nkv, ctx, hd), np.float32)
    g0 = orc.kv_head_of(0, nq, nkv)
    qh = q[0].astype(np.float64)
    kc[g0] = (target / scale)[:, None] * (qh / (qh @ qh))[None, :]
    for g in range(nkv):
        if g != g0:
            kc[g] = rng.normal(0, 1, (ctx, hd))
    kc = _bf16(kc)
    vc = _bf16(rng.normal(0, 1, (nkv, ctx, hd)))
    # the construction, on the stored keys: within a period each chunk's top
    # score is more than the slack above the previous chunk's
    k64 = torch.from_numpy(kc.view(np.int16)).view(torch.bfloat16).double().numpy()
    top = ((k64[g0, :n] @ qh) * scale)[: (n // ch) * ch].reshape(-1, ch).max(axis=1)
    steps = np.diff(top)[(np.arange(len(top) - 1) + 1) % 8 != 0]
    assert steps.min() > 8.0
    kc_dev = torch.from_numpy(kc.view(np.int16)).cuda()
    vc_dev = torch.from_numpy(vc.view(np.int16)).cuda()
    o_dev = torch.full((nq * hd,), float("nan"), device="cuda")
    dec.attention_noalloc(torch.from_numpy(q.ravel()).cuda(), kc_dev, vc_dev, nq, nkv, hd, ctx, n, o_dev)
    dec.noalloc_sync_status()
    got = o_dev.cpu().numpy().reshape(nq, hd)
    for h in range(nq):
        g = orc.kv_head_of(h, nq, nkv)
        ref = orc.attention_head(q[h].astype(np.float64), kc[g, :n], vc[g, :n])
        assert_close(got[h], ref, f"rising scores, hd {hd}, head {h}", max_abs=1e-4, rel_l2=1e-5)
