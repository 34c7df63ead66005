"""Seeded synthetic workloads for the batch-1 decode layer.

The five workloads are Llama-style decoder stacks run one token at a time with a
prefilled KV cache.  Every tensor is drawn from a counter-based generator
(``synth.c``) keyed by (seed, layer, tensor id, element index), so any element
can be regenerated on its own and both the CPU oracle and the CUDA path see the
same bits.  This module only draws and stores numbers; it contains none of the
layer's arithmetic.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass, replace

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libsynth.so")

# tensor ids of the generator key (weights use the ABI's [out][in] orientation)
T_ATTN_NORM, T_WQ, T_WK, T_WV, T_WO, T_FFN_NORM, T_WGATE, T_WUP, T_WDOWN = range(9)
T_KCACHE, T_VCACHE, T_INPUT = 9, 10, 11
T_LM_NORM, T_LM_HEAD = 12, 13  # after the stack (generator layer index -1)
Q4_QUANT_OFFSET, Q4_SCALE_OFFSET = 100, 200
KV_POS_STRIDE = 1 << 24  # element index of K[g][t][i] = (g*KV_POS_STRIDE + t)*d + i

MATRIX_TENSORS = (T_WQ, T_WK, T_WV, T_WO, T_WGATE, T_WUP, T_WDOWN)
NORM_TENSORS = (T_ATTN_NORM, T_FFN_NORM)


@dataclass(frozen=True)
class Workload:
    """One decode workload: model shape, prefilled context and step count."""

    name: str
    n_layers: int
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    prefill: int          # KV positions already in the cache before step 0
    steps: int            # consecutive decode steps from pos = prefill
    weight_fmt: str = "bf16"   # "bf16" or "q4" (int4 per 32 + fp16 scale)
    rms_eps: float = 1e-6
    rope_theta: float = 1e4
    rope_interleaved: bool = False  # RoPE pairs (2i, 2i+1) instead of (i, i + d/2)
    seed: int = 0
    w_std: float = 0.02
    norm_std: float = 0.1
    kv_std: float = 1.0
    q4_scale_std: float = 0.002

    def shape(self, tensor: int) -> tuple[int, int]:
        """[out][in] of a weight matrix."""
        H, d, F = self.hidden, self.head_dim, self.ffn
        return {
            T_WQ: (self.n_q_heads * d, H),
            T_WK: (self.n_kv_heads * d, H),
            T_WV: (self.n_kv_heads * d, H),
            T_WO: (H, self.n_q_heads * d),
            T_WGATE: (F, H),
            T_WUP: (F, H),
            T_WDOWN: (H, F),
        }[tensor]

    def weight_bytes_per_layer(self) -> int:
        n = sum(o * i for o, i in (self.shape(t) for t in MATRIX_TENSORS))
        per = 2.0 if self.weight_fmt == "bf16" else 0.5 + 2.0 / 32
        return int(n * per) + 2 * 2 * self.hidden

    def small(self, **kw) -> "Workload":
        return replace(self, **kw)


# The workloads: one layer at hidden 512; a 1B-shape 16-layer stack; the
# 7B-shape 32-layer MHA stack; a 9B-shape 40-layer GQA stack; the 7B shape with
# int4 weights and int8 activations.
WORKLOADS = {
    "layer_h512": Workload("layer_h512", 1, 512, 8, 2, 64, 1408, prefill=127, steps=1),
    "stack16_h2048": Workload("stack16_h2048", 16, 2048, 32, 8, 64, 8192, prefill=1023, steps=64),
    "stack32_h4096_mha": Workload("stack32_h4096_mha", 32, 4096, 32, 32, 128, 11008,
                                  prefill=2047, steps=128),
    "stack40_h4096_gqa": Workload("stack40_h4096_gqa", 40, 4096, 32, 8, 128, 12288,
                                  prefill=4095, steps=128),
    "stack32_h4096_q4": Workload("stack32_h4096_q4", 32, 4096, 32, 32, 128, 11008,
                                 prefill=2047, steps=128, weight_fmt="q4"),
}

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile synth.c into a shared library next to it (gcc, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".{os.getpid()}.tmp"
        subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"],
                       check=True)
        os.replace(tmp, _SO)
    return _SO


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            u64, i64, dbl, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
            L.synth_splitmix64.restype = u64
            L.synth_splitmix64.argtypes = [u64]
            L.synth_key.restype = u64
            L.synth_key.argtypes = [u64, i64, i64]
            L.synth_round_bf16.restype = ctypes.c_uint16
            L.synth_round_bf16.argtypes = [dbl]
            L.synth_round_fp16.restype = ctypes.c_uint16
            L.synth_round_fp16.argtypes = [dbl]
            for fn in (L.synth_normal_bf16, L.synth_normal_bf16_as_f32, L.synth_absnormal_fp16):
                fn.restype = None
                fn.argtypes = [u64, i64, i64, u64, u64, dbl, dbl, vp]
            L.synth_q4_packed.restype = None
            L.synth_q4_packed.argtypes = [u64, i64, i64, u64, u64, vp]
            _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags.c_contiguous
    return a.ctypes.data


def normal_bf16(seed, layer, tensor, start, count, mean, std) -> np.ndarray:
    out = np.empty(count, dtype=np.uint16)
    lib().synth_normal_bf16(seed, layer, tensor, start, count, mean, std, _ptr(out))
    return out


def weight_bf16(w: Workload, layer: int, tensor: int, out: np.ndarray | None = None) -> np.ndarray:
    """bf16 bits of a [out][in] weight matrix, ~N(0, w_std)."""
    o, i = w.shape(tensor)
    if out is None:
        out = np.empty((o, i), dtype=np.uint16)
    lib().synth_normal_bf16(w.seed, layer, tensor, 0, o * i, 0.0, w.w_std, _ptr(out))
    return out


def norm_bf16(w: Workload, layer: int, tensor: int) -> np.ndarray:
    """bf16 bits of an RMSNorm weight vector, ~1 + N(0, norm_std)."""
    out = np.empty(w.hidden, dtype=np.uint16)
    lib().synth_normal_bf16(w.seed, layer, tensor, 0, w.hidden, 1.0, w.norm_std, _ptr(out))
    return out


def weight_q4(w: Workload, layer: int, tensor: int) -> tuple[np.ndarray, np.ndarray]:
    """(packed int4 [out][in/2] uint8, fp16 scale bits [out][in/32] uint16)."""
    o, i = w.shape(tensor)
    assert i % 32 == 0
    q = np.empty((o, i // 2), dtype=np.uint8)
    lib().synth_q4_packed(w.seed, layer, tensor + Q4_QUANT_OFFSET, o, i, _ptr(q))
    s = np.empty((o, i // 32), dtype=np.uint16)
    lib().synth_absnormal_fp16(w.seed, layer, tensor + Q4_SCALE_OFFSET, 0, o * (i // 32), 0.0,
                               w.q4_scale_std, _ptr(s))
    return q, s


def kv_bf16(w: Workload, layer: int, n_pos: int) -> tuple[np.ndarray, np.ndarray]:
    """Prefilled cache rows: (K, V) bf16 bits, each [n_kv_heads][n_pos][head_dim], ~N(0, kv_std)."""
    d, G = w.head_dim, w.n_kv_heads
    out = []
    for t in (T_KCACHE, T_VCACHE):
        a = np.empty((G, n_pos, d), dtype=np.uint16)
        for g in range(G):
            lib().synth_normal_bf16(w.seed, layer, t, g * KV_POS_STRIDE * d, n_pos * d, 0.0,
                                    w.kv_std, _ptr(a[g]))
        out.append(a)
    return out[0], out[1]


def step_input(w: Workload, step: int) -> np.ndarray:
    """Input hidden vector of decode step `step`: N(0,1) rounded to bf16, as fp32."""
    out = np.empty(w.hidden, dtype=np.float32)
    lib().synth_normal_bf16_as_f32(w.seed, step, T_INPUT, 0, w.hidden, 0.0, 1.0, _ptr(out))
    return out


def lm_head(w: Workload, vocab: int) -> tuple[np.ndarray, np.ndarray]:
    """The LM head after the stack: (final RMSNorm weight bf16 bits [H] ~1 + N(0,
    norm_std), vocabulary matrix bf16 bits [vocab][H] ~N(0, w_std))."""
    nw = np.empty(w.hidden, dtype=np.uint16)
    lib().synth_normal_bf16(w.seed, -1, T_LM_NORM, 0, w.hidden, 1.0, w.norm_std, _ptr(nw))
    W = np.empty((vocab, w.hidden), dtype=np.uint16)
    lib().synth_normal_bf16(w.seed, -1, T_LM_HEAD, 0, vocab * w.hidden, 0.0, w.w_std, _ptr(W))
    return nw, W


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def fp16_to_f32(bits: np.ndarray) -> np.ndarray:
    return bits.view(np.float16).astype(np.float32)


@dataclass
class LayerWeights:
    attn_norm: np.ndarray
    ffn_norm: np.ndarray
    mats: dict            # tensor id -> bf16 bits [out][in]   (bf16 workloads)
    q4: dict              # tensor id -> (packed, scales)      (q4 workloads)


def layer_weights(w: Workload, layer: int) -> LayerWeights:
    mats, q4 = {}, {}
    for t in MATRIX_TENSORS:
        if w.weight_fmt == "bf16":
            mats[t] = weight_bf16(w, layer, t)
        else:
            q4[t] = weight_q4(w, layer, t)
    return LayerWeights(norm_bf16(w, layer, T_ATTN_NORM), norm_bf16(w, layer, T_FFN_NORM), mats, q4)
