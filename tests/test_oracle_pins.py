"""Pins of the fp64 oracle against things other than itself.

Closed forms, invariants, brute force on tiny inputs and special cases that
reduce to library routines (numpy matmul, torch float64 rms_norm / SDPA / silu,
complex multiplication).  Each ``pin_*`` function raises AssertionError on a
mismatch; ``test_planted_mistakes_are_caught`` plants each known mistake in the
oracle and checks that at least one pin fails.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(1234)


def _bf16_bits_from_f32(a: np.ndarray) -> np.ndarray:
    """bf16 bits of float32 values via torch's float32 -> bfloat16 (RNE) cast."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _bf16_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _rand_bf16(shape, std=1.0, mean=0.0):
    return _bf16_bits_from_f32(RNG.normal(mean, std, size=shape).astype(np.float32))


ONE_BF16 = 0x3F80


def _close(a, b, tol=1e-12, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    err = np.max(np.abs(a - b)) if a.size else 0.0
    scale = max(1.0, float(np.max(np.abs(b))) if b.size else 1.0)
    assert err <= tol * scale, f"{what}: max err {err:.3e} > {tol:.1e}*{scale:.3g}"


# ---- storage formats ------------------------------------------------------------

def pin_storage_formats():
    g = json.load(open(os.path.join(GOLDEN, "storage_formats.json")))
    for c in g["bf16_round"]:
        assert orc.bf16_round(c["value"]) == int(c["bits"], 16), c
        assert orc.bf16_value(int(c["bits"], 16)) == orc.bf16_value(orc.bf16_round(c["value"]))
    for c in g["fp16_value"]:
        assert orc.fp16_value(int(c["bits"], 16)) == c["value"], c
    # agrees with torch's float32 -> bfloat16 cast on float32-representable inputs
    x = RNG.normal(0, 3, 2000).astype(np.float32)
    ref = _bf16_bits_from_f32(x)
    mine = np.array([orc.bf16_round(float(v)) for v in x], dtype=np.uint16)
    assert np.array_equal(ref, mine)
    # binary16 decode agrees with numpy's float16 on every finite pattern
    bits = np.arange(0, 0x7C00, 37, dtype=np.uint16)
    ref16 = bits.view(np.float16).astype(np.float64)
    assert all(orc.fp16_value(int(b)) == r for b, r in zip(bits, ref16))


# ---- RMSNorm ---------------------------------------------------------------------

def pin_rmsnorm():
    H = 96
    x = RNG.normal(0, 2, H)
    ones = np.full(H, ONE_BF16, np.uint16)
    eps = 1e-6
    n = orc.rmsnorm(x, ones, eps)
    ms = np.mean(x * x)
    # unit RMS before the weight: mean(n^2) = ms / (ms + eps)
    _close(np.mean(n * n), ms / (ms + eps), 1e-13, "unit rms")
    # scale invariance (exact with eps = 0)
    _close(orc.rmsnorm(7.5 * x, ones, 0.0), orc.rmsnorm(x, ones, 0.0), 1e-13, "scale inv")
    # constant vector, large eps: n = c / sqrt(c^2 + eps) * w
    w = _rand_bf16(H, 0.1, 1.0)
    c, big_eps = -0.5, 0.75
    got = orc.rmsnorm(np.full(H, c), w, big_eps)
    _close(got, c / math.sqrt(c * c + big_eps) * _bf16_f64(w), 1e-13, "constant")
    # library: torch.nn.functional.rms_norm in float64
    ref = F.rms_norm(torch.from_numpy(x), (H,), weight=torch.from_numpy(_bf16_f64(w)), eps=eps)
    _close(orc.rmsnorm(x, w, eps), ref.numpy(), 1e-13, "torch rms_norm")


# ---- GEMV ------------------------------------------------------------------------

def pin_gemv():
    K = 48
    x = RNG.normal(0, 1, K)
    eye = np.where(np.eye(K, dtype=bool), ONE_BF16, 0).astype(np.uint16)
    _close(orc.gemv_bf16(eye, x), x, 0, "identity")
    perm = RNG.permutation(K)
    P = np.zeros((K, K), np.uint16)
    P[np.arange(K), perm] = ONE_BF16
    _close(orc.gemv_bf16(P, x), x[perm], 0, "permutation")
    W = _rand_bf16((40, K), 0.02)
    e = np.zeros(K)
    e[17] = 1.0
    _close(orc.gemv_bf16(W, e), _bf16_f64(W)[:, 17], 0, "one-hot column")
    Wsq = _rand_bf16((K, K), 0.02)       # square and non-symmetric
    _close(orc.gemv_bf16(Wsq, x), _bf16_f64(Wsq) @ x, 1e-13, "numpy matmul (square)")
    _close(orc.gemv_bf16(W, x), _bf16_f64(W) @ x, 1e-13, "numpy matmul")


# ---- RoPE ------------------------------------------------------------------------

def _rope_complex(h, pos, theta):
    """Rotate-half RoPE as complex multiplication (a different formulation)."""
    t = torch.from_numpy(np.asarray(h, dtype=np.float64))
    d = t.shape[-1]
    z = torch.complex(t[..., : d // 2], t[..., d // 2:])
    ang = pos * theta ** (-2.0 * torch.arange(d // 2, dtype=torch.float64) / d)
    z = z * torch.polar(torch.ones_like(ang), ang)
    return torch.cat([z.real, z.imag], dim=-1).numpy()


def pin_rope():
    theta = 1e4
    g = json.load(open(os.path.join(GOLDEN, "rope_closed_forms.json")))
    env = {"cos": math.cos, "sin": math.sin}
    for c in g["cases"]:
        h = np.array(c["h"], dtype=np.float64)[None, :]
        exp = np.array([eval(s, env) for s in c["expected"]])  # closed-form strings
        _close(orc.rope(h, c["pos"], c["theta"])[0], exp, 1e-12, c["name"])
    h = RNG.normal(0, 1, (3, 64))
    _close(orc.rope(h, 0, theta), h, 0, "pos 0 identity")
    r = orc.rope(h, 777, theta)
    pair = lambda v: v[:, :32] ** 2 + v[:, 32:] ** 2
    _close(pair(r), pair(h), 1e-12, "pair norms")
    _close(orc.rope(orc.rope(h, 300, theta), 477, theta), r, 1e-11, "R(a)R(b)=R(a+b)")
    q, k = RNG.normal(0, 1, (1, 64)), RNG.normal(0, 1, (1, 64))
    lhs = float(orc.rope(q, 1000, theta)[0] @ orc.rope(k, 1234, theta)[0])
    rhs = float(q[0] @ orc.rope(k, 234, theta)[0])
    assert abs(lhs - rhs) < 1e-10, ("relative position", lhs, rhs)
    _close(r, _rope_complex(h, 777, theta), 1e-12, "complex formulation")


def pin_rope_interleaved():
    """Interleaved pairs (2i, 2i+1): the rotate-half rotation conjugated by the
    permutation that takes dim 2i to i and 2i+1 to i + d/2; a d = 2 head turns
    by pos radians; identity at pos 0; pair norms kept; and a whole layer with
    interleaved RoPE equals the rotate-half layer on weights whose q/k rows are
    permuted the same way (attention is invariant under a shared permutation of
    q and k dims)."""
    theta, d = 1e4, 64
    perm = np.concatenate([np.arange(0, d, 2), np.arange(1, d, 2)])  # new order of old dims
    h = RNG.normal(0, 1, (3, d))
    got = orc.rope(h, 321, theta, interleaved=True)
    via = np.empty_like(h)
    via[:, perm] = orc.rope(h[:, perm], 321, theta)
    _close(got, via, 1e-12, "interleaved = conjugated rotate-half")
    _close(orc.rope(h, 0, theta, interleaved=True), h, 0, "pos 0 identity")
    pn = lambda v: v[:, 0::2] ** 2 + v[:, 1::2] ** 2
    _close(pn(got), pn(h), 1e-12, "pair norms")
    e = np.array([[1.0, 0.0]])
    _close(orc.rope(e, 3, theta, interleaved=True), np.array([[math.cos(3), math.sin(3)]]), 1e-15,
           "d = 2 turns by pos radians")
    # a layer: interleaved pairs on permuted q/k rows == rotate-half on the originals
    H, nq, nkv, dd, Fd = 32, 2, 1, 8, 48
    lw = _toy_layer(H, nq, nkv, dd, Fd)
    pr = np.concatenate([np.arange(0, dd, 2), np.arange(1, dd, 2)])
    lw_i = dict(lw)
    lw_i["w"] = list(lw["w"])
    for t, heads in ((0, nq), (1, nkv)):
        rows = np.concatenate([hh * dd + np.argsort(pr) for hh in range(heads)])
        lw_i["w"][t] = lw["w"][t][rows]
    kw = dict(hidden=H, n_q_heads=nq, n_kv_heads=nkv, head_dim=dd, ffn=Fd, max_ctx=4)
    a = orc.OracleStack(layers=[lw], **kw)
    b = orc.OracleStack(layers=[lw_i], rope_interleaved=True, **kw)
    for pos in range(3):
        x = RNG.normal(0, 1, H)
        _close(b.step(x, pos), a.step(x, pos), 1e-12, f"interleaved layer, pos {pos}")


# ---- attention -------------------------------------------------------------------

def pin_attention():
    d = 16
    q = RNG.normal(0, 1, d)
    K1, V1 = _rand_bf16((1, d)), _rand_bf16((1, d))
    _close(orc.attention_head(q, K1, V1), _bf16_f64(V1)[0], 1e-15, "n=1 returns v")
    n = 9
    Keq = np.repeat(_rand_bf16((1, d)), n, axis=0)
    V = _rand_bf16((n, d))
    _close(orc.attention_head(q, Keq, V), _bf16_f64(V).mean(0), 1e-14, "equal keys -> mean V")
    # one key far ahead of the rest: o -> that v (the last row, the new token)
    Kd = _bf16_bits_from_f32(np.zeros((n, d), np.float32))
    qd = np.zeros(d)
    qd[0] = 1.0
    Kd[-1, 0] = _bf16_bits_from_f32(np.array([200.0], np.float32))[0]
    _close(orc.attention_head(qd, Kd, V), _bf16_f64(V)[-1], 1e-12, "dominant score")
    # softmax is shift invariant: scores near 1000 (exp overflows in fp64 past
    # ~709) give exactly the output of the same scores moved near 0; keys
    # 2000 + 16 j and 16 j are exact in bf16, q = 2 e0, scale 1/4: scores
    # 1000 + 8 j and 8 j
    Kb = _rand_bf16((n, d))
    Ks = Kb.copy()
    js = np.array([3, 0, 7, 5, 1, 6, 2, 4, 7])
    Kb[:, 0] = _bf16_bits_from_f32((16.0 * js).astype(np.float32))
    Ks[:, 0] = _bf16_bits_from_f32((2000.0 + 16.0 * js).astype(np.float32))
    assert np.all(_bf16_f64(Ks)[:, 0] - _bf16_f64(Kb)[:, 0] == 2000.0)
    q2 = 2.0 * qd
    base = orc.attention_head(q2, Kb, V)
    _close(orc.attention_head(q2, Ks, V), base, 1e-12, "shift invariance at scores ~1000")
    w = np.exp(8.0 * js - 8.0 * js.max())
    _close(base, (w / w.sum()) @ _bf16_f64(V), 1e-12, "softmax weights of the small scores")
    # library: torch SDPA (float64) with GQA
    nq, nkv, n = 8, 2, 23
    Q = RNG.normal(0, 1, (nq, d))
    Kb, Vb = _rand_bf16((nkv, n, d)), _rand_bf16((nkv, n, d))
    ref = F.scaled_dot_product_attention(
        torch.from_numpy(Q)[None, :, None, :], torch.from_numpy(_bf16_f64(Kb))[None],
        torch.from_numpy(_bf16_f64(Vb))[None], enable_gqa=True)[0, :, 0, :].numpy()
    got = np.stack([orc.attention_head(Q[h], Kb[orc.kv_head_of(h, nq, nkv)],
                                       Vb[orc.kv_head_of(h, nq, nkv)]) for h in range(nq)])
    _close(got, ref, 1e-13, "torch SDPA gqa")


# ---- SwiGLU ----------------------------------------------------------------------

def pin_swiglu():
    assert orc.silu(0.0) == 0.0
    assert abs(orc.silu(40.0) - 40.0) < 1e-15 * 40 + 40 * math.exp(-40)
    assert abs(orc.silu(-40.0)) < 1e-15
    g, u = RNG.normal(0, 2, 64), RNG.normal(0, 2, 64)
    ref = (F.silu(torch.from_numpy(g)) * torch.from_numpy(u)).numpy()
    _close(orc.swiglu(g, u), ref, 1e-14, "torch silu(g)*u")


# ---- int4 weights / int8 activations ---------------------------------------------

def pin_quant():
    g = json.load(open(os.path.join(GOLDEN, "quant_examples.json")))
    for c in g["cases"]:
        z = np.full(32, c["z_tail_fill"])
        z[: len(c["z_head"])] = c["z_head"]
        q, dx = orc.quantize_act(z)
        assert float(dx[0]) == c["dx"], (c["name"], dx[0])
        assert list(q[: len(c["q_head"])]) == c["q_head"], (c["name"], q[:8])
    z = RNG.normal(0, 1.5, 256)
    q, dx = orc.quantize_act(z)
    for b in range(8):
        blk = z[32 * b: 32 * b + 32]
        assert abs(int(q[32 * b + np.argmax(np.abs(blk))])) == 127
        assert np.all(np.abs(q[32 * b: 32 * b + 32] * np.float64(dx[b]) - blk) <= dx[b] * 0.5001)


def _pack_q4(qw: np.ndarray) -> np.ndarray:
    u = (qw + 8).astype(np.uint8)
    return (u[:, 0::2] | (u[:, 1::2] << 4)).astype(np.uint8)


def pin_q4_dots():
    N, K = 5, 96
    qw = RNG.integers(-8, 8, (N, K))
    qx = RNG.integers(-127, 128, K).astype(np.int8)
    pk = _pack_q4(qw)
    dots = orc.q4_blockdots(pk, qx)
    for j in range(N):                       # brute force in Python integers
        for b in range(K // 32):
            s = sum(int(qw[j, 32 * b + i]) * int(qx[32 * b + i]) for i in range(32))
            assert dots[j, b] == s
    # scale 1, dx 1: float result is the exact integer sum
    ones = np.full((N, K // 32), 0x3C00, np.uint16)
    y = orc.gemv_q4(pk, ones, qx, np.ones(K // 32, np.float32))
    assert np.array_equal(y, (qw @ qx.astype(np.int64)).astype(np.float64))
    # library: dequantised numpy matmul
    sc = RNG.integers(0x1000, 0x2400, (N, K // 32)).astype(np.uint16)
    dx = np.abs(RNG.normal(0, 0.01, K // 32)).astype(np.float32)
    Wd = qw * np.repeat(sc.view(np.float16).astype(np.float64), 32, axis=1)
    xd = qx * np.repeat(dx.astype(np.float64), 32)
    _close(orc.gemv_q4(pk, sc, qx, dx), Wd @ xd, 1e-13, "dequantised matmul")


# ---- LM head and greedy choice ------------------------------------------------------

def pin_lm_head():
    """A one-hot hidden state picks one column of W: the token is the row whose
    entry in that column is largest (checked against numpy on the column);
    equal largest logits go to the lowest index; the logits equal torch's
    float64 rms_norm followed by numpy's matmul."""
    H, V, eps = 64, 40, 1e-6
    W = _rand_bf16((V, H), 0.5)
    nw = _rand_bf16(H, 0.1, 1.0)
    k = 23
    x = np.zeros(H)
    x[k] = 3.0
    tok, logits = orc.lm_head(x, nw, W, eps)
    col = _bf16_f64(W)[:, k] * _bf16_f64(nw)[k]
    assert tok == int(np.argmax(col)), (tok, int(np.argmax(col)))
    # ties: rows 7 and 19 equal and the largest
    Wt = W.copy()
    Wt[19] = Wt[7]
    top = _bf16_bits_from_f32(np.array([9.0], np.float32))[0]
    Wt[7, k] = Wt[19, k] = top
    assert orc.lm_head(x, nw, Wt, eps)[0] == 7
    # library restatement of the logits
    xr = RNG.normal(0, 2, H)
    n = F.rms_norm(torch.from_numpy(xr), (H,), weight=torch.from_numpy(_bf16_f64(nw)), eps=eps)
    tok, logits = orc.lm_head(xr, nw, W, eps)
    ref = _bf16_f64(W) @ n.numpy()
    _close(logits, ref, 1e-13, "LM head logits")
    assert tok == int(np.argmax(ref))


# ---- whole layer -----------------------------------------------------------------

def _torch_layer(x, lw, pos, theta, eps, Kc, Vc, nq, nkv, d):
    """Float64 torch restatement of one layer from library routines."""
    T = lambda a: torch.from_numpy(np.asarray(a, dtype=np.float64))
    W = [T(_bf16_f64(w)) for w in lw["w"]]
    x = T(x)
    H = x.shape[0]
    n1 = F.rms_norm(x, (H,), weight=T(_bf16_f64(lw["attn_norm"])), eps=eps)
    q, k, v = W[0] @ n1, W[1] @ n1, W[2] @ n1
    q = T(_rope_complex(q.view(nq, d).numpy(), pos, theta))
    k = T(_rope_complex(k.view(nkv, d).numpy(), pos, theta))
    kb = k.to(torch.float32).to(torch.bfloat16).to(torch.float64)
    vb = v.view(nkv, d).to(torch.float32).to(torch.bfloat16).to(torch.float64)
    Kc = Kc.clone()
    Vc = Vc.clone()
    Kc[:, pos] = kb
    Vc[:, pos] = vb
    o = F.scaled_dot_product_attention(q[None, :, None, :], Kc[None, :, : pos + 1],
                                       Vc[None, :, : pos + 1], enable_gqa=True)[0, :, 0, :]
    h1 = x + W[3] @ o.reshape(-1)
    n2 = F.rms_norm(h1, (H,), weight=T(_bf16_f64(lw["ffn_norm"])), eps=eps)
    a = F.silu(W[4] @ n2) * (W[5] @ n2)
    return (h1 + W[6] @ a).numpy(), Kc, Vc


def _toy_layer(H, nq, nkv, d, Fd):
    shapes = [(nq * d, H), (nkv * d, H), (nkv * d, H), (H, nq * d), (Fd, H), (Fd, H), (H, Fd)]
    return dict(attn_norm=_rand_bf16(H, 0.1, 1.0), ffn_norm=_rand_bf16(H, 0.1, 1.0),
                w=[_rand_bf16(s, 0.3 if H <= 16 else 0.05) for s in shapes])


def _check_layer_vs_torch(H, nq, nkv, d, Fd, prefill, steps):
    theta, eps, max_ctx = 1e4, 1e-6, prefill + steps + 3
    lw = _toy_layer(H, nq, nkv, d, Fd)
    st = orc.OracleStack(hidden=H, n_q_heads=nq, n_kv_heads=nkv, head_dim=d, ffn=Fd,
                         max_ctx=max_ctx, layers=[lw], rms_eps=eps, rope_theta=theta)
    Kp, Vp = _rand_bf16((nkv, prefill, d)), _rand_bf16((nkv, prefill, d))
    if prefill:
        st.load_kv(0, Kp, Vp)
    Kc = torch.zeros(nkv, max_ctx, d, dtype=torch.float64)
    Vc = torch.zeros_like(Kc)
    Kc[:, :prefill] = torch.from_numpy(_bf16_f64(Kp))
    Vc[:, :prefill] = torch.from_numpy(_bf16_f64(Vp))
    for s in range(steps):
        x = RNG.normal(0, 1, H)
        pos = prefill + s
        got = st.step(x, pos)
        ref, Kc, Vc = _torch_layer(x, lw, pos, theta, eps, Kc, Vc, nq, nkv, d)
        _close(got, ref, 1e-11, f"layer H={H} pos={pos}")
        # KV append: row pos holds bf16(k_rot), bf16(v); rows past it untouched
        assert np.array_equal(_bf16_f64(st.kcache[0, :, pos]), Kc[:, pos].numpy())
        assert np.array_equal(_bf16_f64(st.vcache[0, :, pos]), Vc[:, pos].numpy())
        assert not st.kcache[0, :, pos + 1:].any()


def pin_layer():
    _check_layer_vs_torch(8, 2, 1, 4, 16, prefill=0, steps=3)      # hidden-8 toy
    _check_layer_vs_torch(64, 4, 2, 16, 96, prefill=5, steps=2)    # GQA 2:1
    _check_layer_vs_torch(64, 8, 2, 8, 64, prefill=7, steps=2)     # GQA 4:1
    _check_layer_vs_torch(32, 2, 2, 16, 48, prefill=3, steps=1)    # MHA


def pin_residual_wiring():
    H, nq, nkv, d, Fd = 32, 4, 2, 8, 48
    lw = _toy_layer(H, nq, nkv, d, Fd)
    lw["w"][3] = np.zeros_like(lw["w"][3])
    lw["w"][6] = np.zeros_like(lw["w"][6])
    st = orc.OracleStack(hidden=H, n_q_heads=nq, n_kv_heads=nkv, head_dim=d, ffn=Fd,
                         max_ctx=4, layers=[lw, lw])
    x = RNG.normal(0, 1, H)
    assert np.array_equal(st.step(x, 0), x)


def pin_kv_append_closed_form():
    # pos 0 (RoPE is the identity), unit norm weights, Wk/Wv pick coordinates:
    # x = +-1 so mean(x^2) = 1 and k_i = x_i / sqrt(1 + eps).
    H, nq, nkv, d, Fd, eps = 16, 2, 2, 4, 16, 0.25
    lw = _toy_layer(H, nq, nkv, d, Fd)
    lw["attn_norm"] = np.full(H, ONE_BF16, np.uint16)
    sel = np.zeros((nkv * d, H), np.uint16)
    sel[np.arange(nkv * d), np.arange(nkv * d)] = ONE_BF16
    lw["w"][1] = sel
    lw["w"][2] = sel[::-1].copy()
    st = orc.OracleStack(hidden=H, n_q_heads=nq, n_kv_heads=nkv, head_dim=d, ffn=Fd,
                         max_ctx=3, layers=[lw], rms_eps=eps)
    st.kcache[...] = 0xABCD        # canaries
    st.vcache[...] = 0xABCD
    x = np.where(RNG.random(H) < 0.5, -1.0, 1.0)
    st.step(x, 0)
    r = 1.0 / math.sqrt(1.0 + eps)
    kexp = np.array([orc.bf16_round(v) for v in x[: nkv * d] * r], np.uint16).reshape(nkv, d)
    vexp = np.array([orc.bf16_round(v) for v in x[: nkv * d][::-1] * r], np.uint16).reshape(nkv, d)
    assert np.array_equal(st.kcache[0, :, 0], kexp)
    assert np.array_equal(st.vcache[0, :, 0], vexp)
    assert np.all(st.kcache[0, :, 1:] == 0xABCD) and np.all(st.vcache[0, :, 1:] == 0xABCD)
    # the bf16 of x/sqrt(1.25) by hand: 1/sqrt(1.25) = 0.894427..., bf16 -> 0.89453125
    assert orc.bf16_value(orc.bf16_round(r)) == 0.89453125
    # the fp64 k, v before the storage rounding come out and round to the row;
    # with the row handed in, the layer leaves it as it is and attends to it
    out, (kz, vz) = st.layer_step(0, x, 0, kvz=True)
    _close(kz, (x[: nkv * d] * r).reshape(nkv, d), 1e-15, "pre-rounding k")
    _close(vz, (x[: nkv * d][::-1] * r).reshape(nkv, d), 1e-15, "pre-rounding v")
    st.vcache[0, :, 0] = 0
    moved = st.layer_step(0, x, 0, kv_given=True)
    assert np.all(st.vcache[0, :, 0] == 0) and not np.array_equal(moved, out)


def pin_q4_layer():
    """A q4 layer whose weights and activations make the integer path exact."""
    H, nq, nkv, d, Fd = 64, 2, 2, 16, 64
    shapes = [(nq * d, H), (nkv * d, H), (nkv * d, H), (H, nq * d), (Fd, H), (Fd, H), (H, Fd)]
    q4 = []
    deq = []
    for o, i in shapes:
        qw = RNG.integers(-8, 8, (o, i))
        sc = np.full((o, i // 32), 0x2C00, np.uint16)   # fp16 0.0625
        q4.append((_pack_q4(qw), sc))
        deq.append(qw * 0.0625)
    lw = dict(attn_norm=_rand_bf16(H, 0.1, 1.0), ffn_norm=_rand_bf16(H, 0.1, 1.0), q4=q4)
    st = orc.OracleStack(hidden=H, n_q_heads=nq, n_kv_heads=nkv, head_dim=d, ffn=Fd,
                         max_ctx=2, layers=[lw], q4=True)
    x = RNG.normal(0, 1, H)
    out, taps = st.layer_step(0, x, 0, qtap=True)
    # the captured int8 input of the q projection is the quantisation of n1
    n1 = orc.rmsnorm(x, lw["attn_norm"], 1e-6)
    q_ref, d_ref = orc.quantize_act(n1)
    assert np.array_equal(taps[0][0], q_ref) and np.array_equal(taps[0][1], d_ref)
    # and the q4 projection equals the dequantised matmul of the int8 input
    xq = taps[0][0] * np.repeat(taps[0][1].astype(np.float64), 32)
    q_proj = orc.gemv_q4(q4[0][0], q4[0][1], taps[0][0], taps[0][1])
    _close(q_proj, deq[0] @ xq, 1e-13, "q4 projection")
    assert np.all(np.isfinite(out))
    # given codes: its own codes reproduce the layer exactly; one code of the
    # down projection's input raised by one moves output j by exactly
    # scale * dx_b * w[j][k] (the residual and everything before stay put)
    again = st.layer_step(0, x, 0, qgiven=taps)
    assert np.array_equal(again, out)
    # slot by slot: the first slot's own codes given, the rest quantized here,
    # reproduce the layer; each slot's fp64 input vector comes out and
    # quantizes to that slot's codes
    part, trip = st.layer_step(0, x, 0, qgiven=[taps[0], None, None, None], zout=True)
    assert np.array_equal(part, out)
    _close(trip[0][2], n1, 0, "z of the q projection's input")
    for slot in range(4):
        qz, dz = orc.quantize_act(trip[slot][2])
        assert np.array_equal(qz, trip[slot][0]) and np.array_equal(dz, trip[slot][1]), slot
    k = 37
    qa = taps[3][0].copy()
    assert abs(int(qa[k])) < 127
    qa[k] += 1
    moved = st.layer_step(0, x, 0, qgiven=[taps[0], taps[1], taps[2], (qa, taps[3][1])])
    step = 0.0625 * float(taps[3][1][k // 32]) * deq[6][:, k] / 0.0625
    _close(moved - out, step, 1e-9, "one int8 code of the down input")


def pin_layer_brute_force():
    """The hidden-8 toy layer written out as explicit scalar sums in plain Python
    (no matrix routine): two q heads sharing one KV head, head dim 4, FFN 16,
    three decode steps from an empty cache."""
    H, nq, nkv, d, Fd, eps, theta = 8, 2, 1, 4, 16, 1e-6, 1e4
    lw = _toy_layer(H, nq, nkv, d, Fd)
    st = orc.OracleStack(hidden=H, n_q_heads=nq, n_kv_heads=nkv, head_dim=d, ffn=Fd,
                         max_ctx=4, layers=[lw], rms_eps=eps, rope_theta=theta)
    W = [_bf16_f64(w).tolist() for w in lw["w"]]
    g_in, g_post = _bf16_f64(lw["attn_norm"]).tolist(), _bf16_f64(lw["ffn_norm"]).tolist()

    def bf16(v):  # the cache's storage rounding (fp32, then round-to-nearest-even bf16)
        return float(torch.tensor([v], dtype=torch.float32).to(torch.bfloat16).to(torch.float64)[0])

    def rms(v, g):
        ms = 0.0
        for e in v:
            ms += e * e
        r = 1.0 / math.sqrt(ms / len(v) + eps)
        return [v[i] * r * g[i] for i in range(len(v))]

    def mv(M, v):
        out = []
        for row in M:
            acc = 0.0
            for i in range(len(v)):
                acc += row[i] * v[i]
            out.append(acc)
        return out

    def rope(v, pos):
        out = list(v)
        for h in range(len(v) // d):
            for i in range(d // 2):
                ang = pos * theta ** (-2.0 * i / d)
                a, b = v[h * d + i], v[h * d + i + d // 2]
                out[h * d + i] = a * math.cos(ang) - b * math.sin(ang)
                out[h * d + i + d // 2] = a * math.sin(ang) + b * math.cos(ang)
        return out

    Kc, Vc = [], []
    for step in range(3):
        pos = step
        x = RNG.normal(0, 1, H).tolist()
        n1 = rms(x, g_in)
        q, k, v = rope(mv(W[0], n1), pos), rope(mv(W[1], n1), pos), mv(W[2], n1)
        Kc.append([bf16(e) for e in k])
        Vc.append([bf16(e) for e in v])
        o = []
        for h in range(nq):  # both q heads read KV head 0
            s = []
            for t in range(pos + 1):
                dot = 0.0
                for i in range(d):
                    dot += q[h * d + i] * Kc[t][i]
                s.append(dot / math.sqrt(d))
            m = max(s)
            e = [math.exp(z - m) for z in s]
            tot = sum(e)
            for i in range(d):
                acc = 0.0
                for t in range(pos + 1):
                    acc += e[t] / tot * Vc[t][i]
                o.append(acc)
        h1 = [x[i] + y for i, y in enumerate(mv(W[3], o))]
        n2 = rms(h1, g_post)
        gt, up = mv(W[4], n2), mv(W[5], n2)
        a = [gt[j] / (1.0 + math.exp(-gt[j])) * up[j] for j in range(Fd)]
        ref = [h1[i] + y for i, y in enumerate(mv(W[6], a))]
        got = st.step(np.array(x), pos)
        _close(got, np.array(ref), 1e-12, f"hidden-8 brute force, step {step}")


def _quantize_block_py(z):
    """One 32-block of a GEMV input quantized to int8, written from the reading
    (absmax scale in fp32, fp32 quotient, round half to even, clamp to +-127),
    with numpy float32 scalars for the fp32 steps and Python's round (ties to
    even) for the rounding; independent of the oracle's C quantizer."""
    amax = 0.0
    for v in z:
        amax = max(amax, abs(v))
    d = np.float32(np.float32(amax) / np.float32(127.0))
    q = []
    for v in z:
        if d == 0:
            q.append(0)
        else:
            r = round(float(np.float32(np.float32(v) / d)))
            q.append(max(-127, min(127, r)))
    return q, float(d)


def _q4_layer_py(x, lw, pos, Kc, Vc, nq, nkv, d, eps, theta):
    """One int4-weight / int8-activation layer as explicit scalar sums in plain
    Python.  Kc, Vc: the layer's cache rows so far ([nkv] lists of rows of
    floats); this token's k, v rows are appended.  Returns (out, codes) with
    codes the four GEMV inputs' int8 codes (n1, o, n2, a)."""
    H = len(x)

    def deq_mv(packed, scales, z):
        qz, dz = [], []
        for b in range(len(z) // 32):
            qb, db = _quantize_block_py(z[32 * b: 32 * b + 32])
            qz += qb
            dz.append(db)
        out = []
        for j in range(packed.shape[0]):
            acc = 0.0
            for b in range(len(z) // 32):
                idot = 0
                for i in range(32):
                    k = 32 * b + i
                    byte = int(packed[j, k // 2])
                    nib = (byte >> 4) if k % 2 else (byte & 15)
                    idot += (nib - 8) * qz[k]
                sw = float(np.uint16(scales[j, b]).view(np.float16))
                acc += sw * dz[b] * idot
            out.append(acc)
        return out, qz

    def rms(v, g):
        ms = 0.0
        for e in v:
            ms += e * e
        r = 1.0 / math.sqrt(ms / len(v) + eps)
        return [v[i] * r * g[i] for i in range(len(v))]

    def rope(v):
        out = list(v)
        for h in range(len(v) // d):
            for i in range(d // 2):
                ang = pos * theta ** (-2.0 * i / d)
                a, b = v[h * d + i], v[h * d + i + d // 2]
                out[h * d + i] = a * math.cos(ang) - b * math.sin(ang)
                out[h * d + i + d // 2] = a * math.sin(ang) + b * math.cos(ang)
        return out

    def bf16(v):  # cache storage rounding (torch's cast)
        return float(torch.tensor([v], dtype=torch.float64).to(torch.bfloat16).to(torch.float64)[0])

    W = lw["q4"]
    g_in, g_post = _bf16_f64(lw["attn_norm"]).tolist(), _bf16_f64(lw["ffn_norm"]).tolist()
    n1 = rms(x, g_in)
    q, c0 = deq_mv(*W[0], n1)
    k, _ = deq_mv(*W[1], n1)
    v, _ = deq_mv(*W[2], n1)
    q, k = rope(q), rope(k)
    for g in range(nkv):
        Kc[g].append([bf16(e) for e in k[g * d:(g + 1) * d]])
        Vc[g].append([bf16(e) for e in v[g * d:(g + 1) * d]])
    o = []
    for h in range(nq):
        g = h * nkv // nq
        s = []
        for t in range(len(Kc[g])):
            dot = 0.0
            for i in range(d):
                dot += q[h * d + i] * Kc[g][t][i]
            s.append(dot / math.sqrt(d))
        m = max(s)
        e = [math.exp(z - m) for z in s]
        tot = sum(e)
        for i in range(d):
            acc = 0.0
            for t in range(len(s)):
                acc += e[t] / tot * Vc[g][t][i]
            o.append(acc)
    y, c1 = deq_mv(*W[3], o)
    h1 = [x[i] + y[i] for i in range(H)]
    n2 = rms(h1, g_post)
    gt, c2 = deq_mv(*W[4], n2)
    up, _ = deq_mv(*W[5], n2)
    a = [gt[j] / (1.0 + math.exp(-gt[j])) * up[j] for j in range(len(gt))]
    y, c3 = deq_mv(*W[6], a)
    return [h1[i] + y[i] for i in range(H)], (c0, c1, c2, c3)


def _q4_toy_layer(H, nq, nkv, d, Fd, scale_std):
    shapes = [(nq * d, H), (nkv * d, H), (nkv * d, H), (H, nq * d), (Fd, H), (Fd, H), (H, Fd)]
    q4 = []
    for o, i in shapes:
        qw = RNG.integers(-8, 8, (o, i))
        sc = np.abs(RNG.normal(0, scale_std, (o, i // 32))).astype(np.float16).view(np.uint16)
        q4.append((_pack_q4(qw), sc))
    return dict(attn_norm=_rand_bf16(H, 0.1, 1.0), ffn_norm=_rand_bf16(H, 0.1, 1.0), q4=q4)


def pin_q4_layer_restated():
    """Whole int4/int8 layers against the plain-Python restatement above: every
    GEMV input's int8 codes equal and every layer output within 1e-12, over
    consecutive steps with a prefilled cache.  Shapes: o shorter than the hidden
    vector (MHA) and o as long as it (GQA 2), FFN of three and two blocks."""
    for H, nq, nkv, d, Fd, prefill, steps, sstd in ((64, 2, 2, 16, 96, 3, 2, 0.05),
                                                     (96, 4, 2, 16, 64, 0, 2, 0.03)):
        eps, theta = 1e-6, 1e4
        lw = _q4_toy_layer(H, nq, nkv, d, Fd, sstd)
        st = orc.OracleStack(hidden=H, n_q_heads=nq, n_kv_heads=nkv, head_dim=d, ffn=Fd,
                             max_ctx=prefill + steps + 1, layers=[lw], rms_eps=eps,
                             rope_theta=theta, q4=True)
        Kp, Vp = _rand_bf16((nkv, prefill, d)), _rand_bf16((nkv, prefill, d))
        if prefill:
            st.load_kv(0, Kp, Vp)
        Kc = [[list(r) for r in _bf16_f64(Kp[g])] for g in range(nkv)]
        Vc = [[list(r) for r in _bf16_f64(Vp[g])] for g in range(nkv)]
        for s in range(steps):
            pos = prefill + s
            x = RNG.normal(0, 1, H).tolist()
            out, taps = st.layer_step(0, np.array(x), pos, qtap=True)
            ref, codes = _q4_layer_py(x, lw, pos, Kc, Vc, nq, nkv, d, eps, theta)
            for slot in range(4):
                assert np.array_equal(taps[slot][0].astype(np.int64), np.array(codes[slot])), \
                    f"q4 layer H={H} pos={pos}: int8 codes of GEMV input {slot} differ"
            _close(out, np.array(ref), 1e-12, f"q4 layer H={H} pos={pos}")
            st.kv_len = pos + 1


PINS = [pin_storage_formats, pin_rmsnorm, pin_gemv, pin_rope, pin_rope_interleaved,
        pin_attention, pin_swiglu, pin_lm_head,
        pin_quant, pin_q4_dots, pin_layer, pin_residual_wiring, pin_kv_append_closed_form,
        pin_q4_layer, pin_layer_brute_force, pin_q4_layer_restated]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin()


@pytest.mark.parametrize("name", [m for m in orc.MUTATIONS if m != "none"])
def test_planted_mistakes_are_caught(name):
    """Each plausible mistake planted in the oracle makes at least one pin fail."""
    failed = []
    with orc.mutation(name):
        for pin in PINS:
            try:
                pin()
            except AssertionError:
                failed.append(pin.__name__)
    assert failed, f"mutation {name} went unnoticed by every pin"
