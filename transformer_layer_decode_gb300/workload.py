"""Builds a :class:`~.dec.Decoder` for one of the synthetic workloads.

Weights, the prefilled KV cache and the per-step inputs all come from the
seeded generator in :mod:`.synth`; this module only moves them into the
library through its C ABI.
"""
from __future__ import annotations

import numpy as np

from . import dec, synth

_ABI_TENSOR = {
    synth.T_WQ: dec.DEC_T_WQ, synth.T_WK: dec.DEC_T_WK, synth.T_WV: dec.DEC_T_WV,
    synth.T_WO: dec.DEC_T_WO, synth.T_WGATE: dec.DEC_T_WGATE, synth.T_WUP: dec.DEC_T_WUP,
    synth.T_WDOWN: dec.DEC_T_WDOWN,
}


def shape_of(w: synth.Workload, max_ctx: int | None = None) -> dec.Shape:
    if max_ctx is None:
        max_ctx = w.prefill + w.steps + 1
    return dec.Shape(w.n_layers, w.hidden, w.n_q_heads, w.n_kv_heads, w.head_dim, w.ffn, max_ctx,
                     w.rms_eps, w.rope_theta,
                     dec.DEC_W_BF16 if w.weight_fmt == "bf16" else dec.DEC_W_Q4B32)


def load_layer(d: dec.Decoder, w: synth.Workload, layer: int, lw: synth.LayerWeights):
    d.load_weights(layer, dec.DEC_T_ATTN_NORM, lw.attn_norm)
    d.load_weights(layer, dec.DEC_T_FFN_NORM, lw.ffn_norm)
    for t, abi in _ABI_TENSOR.items():
        if w.weight_fmt == "bf16":
            d.load_weights(layer, abi, lw.mats[t])
        else:
            packed, scales = lw.q4[t]
            d.load_weights(layer, abi, packed)
            d.load_weights(layer, abi + dec.DEC_T_SCALES, scales)


def make_decoder(w: synth.Workload, *, max_ctx: int | None = None, unfused: bool = False,
                 graph: bool = True, pdl: bool = True, persistent: bool = False,
                 cluster_attn: bool = True, l2_ahead: bool = True, three: bool = False,
                 four: bool = False, paged_kv: bool = False, page_table=None,
                 q4_publish: bool = False, attn_oproj: bool = False,
                 keep_host: bool = False):
    """Create a decoder with every layer's weights and KV prefill loaded.

    Returns (decoder, host) where host is None or, with keep_host, a dict with
    the per-layer weights and KV prefill arrays (for the CPU oracle)."""
    d = dec.Decoder(shape_of(w, max_ctx), unfused=unfused, graph=graph, pdl=pdl,
                    persistent=persistent, cluster_attn=cluster_attn, l2_ahead=l2_ahead,
                    three=three, four=four, rope_interleaved=w.rope_interleaved,
                    paged_kv=paged_kv, q4_publish=q4_publish,
                    attn_oproj=attn_oproj)
    if page_table is not None:
        d.set_page_table(page_table)
    host = {"layers": [], "kv": []} if keep_host else None
    for layer in range(w.n_layers):
        lw = synth.layer_weights(w, layer)
        load_layer(d, w, layer, lw)
        k, v = synth.kv_bf16(w, layer, w.prefill)
        d.load_kv(layer, k, v, w.prefill)
        if keep_host:
            host["layers"].append(lw)
            host["kv"].append((k, v))
    return d, host


def step_inputs(w: synth.Workload, n: int) -> np.ndarray:
    return np.stack([synth.step_input(w, s) for s in range(n)])
