"""Shared helpers of the parity tests: run a workload on the GPU through the C
ABI and on the fp64 oracle on the same seeded inputs, and compare per layer."""
from __future__ import annotations

import numpy as np

from oracle import oracle as orc
from transformer_layer_decode_gb300 import synth, workload

# Tolerance on every layer's output hidden state (bf16 weights).
MAX_ABS = 2e-2
REL_L2 = 5e-3


def oracle_stack(w: synth.Workload, host: dict, max_ctx: int) -> orc.OracleStack:
    layers = []
    for lw in host["layers"]:
        order = (synth.T_WQ, synth.T_WK, synth.T_WV, synth.T_WO, synth.T_WGATE, synth.T_WUP,
                 synth.T_WDOWN)
        if w.weight_fmt == "bf16":
            layers.append(dict(attn_norm=lw.attn_norm, ffn_norm=lw.ffn_norm,
                               w=[lw.mats[t] for t in order]))
        else:
            layers.append(dict(attn_norm=lw.attn_norm, ffn_norm=lw.ffn_norm,
                               q4=[lw.q4[t] for t in order]))
    st = orc.OracleStack(hidden=w.hidden, n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads,
                         head_dim=w.head_dim, ffn=w.ffn, max_ctx=max_ctx, layers=layers,
                         rms_eps=w.rms_eps, rope_theta=w.rope_theta, q4=w.weight_fmt == "q4")
    for l, (k, v) in enumerate(host["kv"]):
        if w.prefill:
            st.load_kv(l, k, v)
    st.kv_len = w.prefill
    return st


def errors(got: np.ndarray, ref: np.ndarray) -> tuple[float, float]:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    max_abs = float(np.max(np.abs(got - ref)))
    rel = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30))
    return max_abs, rel


def assert_close(got, ref, what: str, max_abs=MAX_ABS, rel_l2=REL_L2):
    a, r = errors(got, ref)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    assert a <= max_abs and r <= rel_l2, f"{what}: max|err| {a:.3e} (<= {max_abs}), rel-L2 {r:.3e} (<= {rel_l2})"
    return a, r


def run_gpu(d, w: synth.Workload, inputs: np.ndarray, *, taps: bool = True):
    """Decode len(inputs) steps from pos = prefill; returns [steps][layers][H] (or [steps][H])."""
    import torch
    dev = torch.device("cuda")
    H, L = w.hidden, w.n_layers
    tap = torch.zeros(L, H, dtype=torch.float32, device=dev) if taps else None
    if taps:
        d.set_tap(tap)
    emb = torch.empty(H, dtype=torch.float32, device=dev)
    out = torch.empty(H, dtype=torch.float32, device=dev)
    res = []
    for s, x in enumerate(inputs):
        emb.copy_(torch.from_numpy(x))
        d.step(emb, w.prefill + s, out)
        d.sync_status()
        res.append((tap if taps else out).cpu().numpy().copy())
    return np.stack(res)


def run_oracle(st: orc.OracleStack, w: synth.Workload, inputs: np.ndarray):
    res = []
    for s, x in enumerate(inputs):
        _, per_layer = st.step(x, w.prefill + s, per_layer=True)
        res.append(per_layer)
    return np.stack(res)


def tiled_rows_to_abi(w: synth.Workload, kernel: int):
    """(tensor id, ABI row) of every tiled row of a fused GEMV, in tiled order:
    QKV rows pair-interleaved per q / k head then v; gate / up rows alternating."""
    hd, nq, nkv = w.head_dim, w.n_q_heads, w.n_kv_heads
    out = []
    if kernel == 0:
        for t, heads in ((synth.T_WQ, nq), (synth.T_WK, nkv)):
            for R in range(heads * hd):
                head, j = divmod(R, hd)
                out.append((t, head * hd + (j // 2 if j % 2 == 0 else j // 2 + hd // 2)))
        out += [(synth.T_WV, r) for r in range(nkv * hd)]
    elif kernel == 3:
        for R in range(2 * w.ffn):
            out.append((synth.T_WGATE if R % 2 == 0 else synth.T_WUP, R // 2))
    else:
        t = synth.T_WO if kernel == 2 else synth.T_WDOWN
        out += [(t, r) for r in range(w.shape(t)[0])]
    return out
