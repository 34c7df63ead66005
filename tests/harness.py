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
                         rms_eps=w.rms_eps, rope_theta=w.rope_theta, q4=w.weight_fmt == "q4",
                         rope_interleaved=w.rope_interleaved)
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


# ---- the int4 / int8 path: integer decisions ---------------------------------

Q4_SLOTS = ("n1 (q/k/v input)", "o (o-proj input)", "n2 (gate/up input)", "a (down input)")


def q4_slot_ks(w: synth.Workload) -> tuple[int, int, int, int]:
    return (w.hidden, w.n_q_heads * w.head_dim, w.hidden, w.ffn)


def bf16_flips(z: np.ndarray, gpu_bits: np.ndarray, rel_tol: float = 1e-5):
    """The GPU's stored bf16 values against the oracle's own rounding of its fp64
    values z ([heads][d]).  Storage rounding decides a discrete value from
    floating point; the GPU rounds its fp32 value, whose arithmetic error is
    absolute (relative to the magnitudes summed, not to the element), so next
    to a rounding midpoint the two may store neighbouring values, and a value
    near zero may differ by more than one bf16 step.  Every difference must
    still be a correct rounding of a value within rel_tol x (the head's RMS)
    of z: |stored - z| <= half the stored value's bf16 step + rel_tol x RMS.
    Returns (number of differing elements, largest excess of |stored - z| over
    its half step, in units of rel_tol x RMS)."""
    z = np.asarray(z, np.float64)
    gpu = np.asarray(gpu_bits, np.uint16).reshape(z.shape)
    own = np.array([orc.bf16_round(float(v)) for v in z.ravel()], np.uint16).reshape(z.shape)
    diff = own != gpu
    if not diff.any():
        return 0, 0.0
    rms = np.sqrt(np.mean(z * z, axis=-1, keepdims=True)) * np.ones_like(z)
    vg = (gpu.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    # the bf16 step at the stored value: 2^(exponent - 7)
    _, e = np.frexp(vg)
    half_step = np.ldexp(1.0, e - 9)
    excess = (np.abs(vg - z) - half_step)[diff] / (rel_tol * rms[diff])
    return int(diff.sum()), float(max(excess.max(), 0.0))


def kv_row_flips(st: orc.OracleStack, layer: int, x, pos: int, k_row: np.ndarray,
                 v_row: np.ndarray):
    """The GPU's appended KV row (bf16 bits [n_kv][d] each) against the oracle's
    own storage rounding of this token's k and v, the layer taking the GPU's
    layer input x; the oracle's cache is left as it is.  Returns (differing
    elements, largest excess over the tolerance of bf16_flips, elements)."""
    _, (kz, vz) = st.layer_step(layer, x, pos, kv_given=True, kvz=True)
    nk, dk = bf16_flips(kz, k_row)
    nv, dv = bf16_flips(vz, v_row)
    return nk + nv, max(dk, dv), kz.size + vz.size


def q4_code_flips(st: orc.OracleStack, w: synth.Workload, layer: int, x, pos: int,
                  gpu_codes: np.ndarray, gpu_scales: np.ndarray, k_row: np.ndarray,
                  v_row: np.ndarray):
    """The GPU's integer decisions of one layer against the oracle's, one at a
    time: the int8 codes of the four GEMV inputs and the bf16 KV row.  For
    slot s the oracle layer takes the GPU's layer input x, the GPU's codes for
    the slots before s and, from slot 1 on, the GPU's appended KV row (so the
    vector it quantizes follows the same decisions) and quantizes slot s itself.
    Where floating point decides an integer the two sides' values differ in
    their last bits, so a code may differ by one where the value sits next to
    a rounding boundary; every difference must be such a flip: |diff| = 1 and
    the oracle's fp32 quotient z/dx within a small distance of a half-integer.

    Returns {"slots": per slot (flips, largest distance of a flip's quotient
    from the half-integer, K), "kv": (flips, largest excess over the tolerance
    of bf16_flips (<= 1 passes), elements)}.  Leaves the GPU's KV row in the
    oracle's cache at pos."""
    Ks = q4_slot_ks(w)
    res = {"slots": []}
    st.kcache[layer, :, pos] = k_row
    st.vcache[layer, :, pos] = v_row
    for s, K in enumerate(Ks):
        given = [(gpu_codes[i, :Ks[i]], gpu_scales[i, :Ks[i] // 32]) if i < s else None
                 for i in range(4)]
        out = st.layer_step(layer, x, pos, qgiven=given, zout=True, kv_given=True, kvz=(s == 1))
        trip = out[1]
        if s == 1:  # this token's k, v from the GPU's n1 codes, before the storage rounding
            kz, vz = out[2]
            nk, dk = bf16_flips(kz, k_row)
            nv, dv = bf16_flips(vz, v_row)
            res["kv"] = (nk + nv, max(dk, dv), kz.size + vz.size)
        own_q, own_d, z = trip[s]
        diff = gpu_codes[s, :K].astype(np.int32) - own_q.astype(np.int32)
        idx = np.nonzero(diff)[0]
        assert np.all(np.abs(diff[idx]) == 1), \
            f"layer {layer} {Q4_SLOTS[s]}: codes differ by more than one"
        quot = z[idx].astype(np.float32) / own_d[idx // 32]
        frac = np.abs(quot.astype(np.float64) - np.trunc(quot.astype(np.float64)))
        dist = float(np.max(np.abs(frac - 0.5))) if idx.size else 0.0
        res["slots"].append((int(idx.size), dist, K))
    return res
