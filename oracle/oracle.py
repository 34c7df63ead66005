"""ctypes front end of the fp64 CPU oracle (oracle.c).

TEST INFRASTRUCTURE ONLY.  Only tests/, ``__graft_entry__.smoke()`` and the
benchmark's cpu_baseline / reference leg may import this module.  It shares no
code with the CUDA library and imports nothing from it.

``OracleStack`` runs the plain unfused decode chain of a Llama-style stack one
token at a time in double precision, with its own bf16 KV cache.  Weights are
passed in as the raw storage arrays (bf16 bits, or packed int4 + fp16 scale
bits) and are read in place.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")

MUTATIONS = {
    "none": 0, "rms_no_eps": 1, "rms_no_weight": 2, "rope_sign": 3, "rope_freq": 4,
    "attn_no_scale": 5, "attn_gqa_mod": 6, "silu_on_up": 7, "no_residual2": 8,
    "gemv_transpose": 9, "q4_no_offset": 10, "attn_skip_last": 11,
    "q4_stale_n1_codes": 12, "q4_o_tensor_scale": 13, "q4_a_no_dx": 14,
    "rope_pair_swap": 15, "argmax_last_tie": 16, "lm_no_norm": 17, "attn_no_max": 18,
}

# Tensor order of the layer struct's matrix slots.
W_Q, W_K, W_V, W_O, W_GATE, W_UP, W_DOWN = range(7)


class Dims(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("n_q_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("ffn", ctypes.c_int32), ("max_ctx", ctypes.c_int32), ("q4", ctypes.c_int32),
                ("rope_interleaved", ctypes.c_int32), ("rms_eps", ctypes.c_double),
                ("rope_theta", ctypes.c_double)]


class Layer(ctypes.Structure):
    _fields_ = [("attn_norm", ctypes.c_void_p), ("ffn_norm", ctypes.c_void_p),
                ("w", ctypes.c_void_p * 7), ("q", ctypes.c_void_p * 7),
                ("s", ctypes.c_void_p * 7), ("kcache", ctypes.c_void_p),
                ("vcache", ctypes.c_void_p)]


class QTap(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p * 4), ("d", ctypes.c_void_p * 4),
                ("z", ctypes.c_void_p * 4), ("kz", ctypes.c_void_p), ("vz", ctypes.c_void_p),
                ("given", ctypes.c_int32), ("kv_given", ctypes.c_int32)]


_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (-O2, OpenMP) into oracle/_build/liboracle.so."""
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
            vp, i32, dbl = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
            sig = {
                "orc_set_mutation": (None, [i32]),
                "orc_get_mutation": (i32, []),
                "orc_bf16_value": (dbl, [ctypes.c_uint16]),
                "orc_fp16_value": (dbl, [ctypes.c_uint16]),
                "orc_bf16_round": (ctypes.c_uint16, [dbl]),
                "orc_rmsnorm": (None, [vp, vp, i32, dbl, vp]),
                "orc_gemv_bf16": (None, [vp, i32, i32, vp, vp]),
                "orc_rope": (None, [vp, i32, i32, i32, dbl]),
                "orc_rope_interleaved": (None, [vp, i32, i32, i32, dbl]),
                "orc_attention_head": (None, [vp, vp, vp, i32, i32, vp]),
                "orc_kv_head_of": (i32, [i32, i32, i32]),
                "orc_silu": (dbl, [dbl]),
                "orc_swiglu": (None, [vp, vp, i32, vp]),
                "orc_quantize_act": (None, [vp, i32, vp, vp]),
                "orc_q4_blockdots": (None, [vp, i32, i32, vp, vp]),
                "orc_gemv_q4": (None, [vp, vp, i32, i32, vp, vp, vp]),
                "orc_layer_step": (i32, [vp, vp, i32, vp, vp, vp]),
                "orc_stack_step": (i32, [vp, vp, i32, i32, vp, vp, vp]),
                "orc_lm_head": (i32, [vp, i32, vp, vp, i32, dbl, vp]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def _p(a: np.ndarray | None) -> int | None:
    if a is None:
        return None
    assert a.flags.c_contiguous, "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _f64(x) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.float64)


class mutation:
    """Context manager planting a known mistake in the oracle (pin tests only)."""

    def __init__(self, name: str):
        self.code = MUTATIONS[name]

    def __enter__(self):
        lib().orc_set_mutation(self.code)

    def __exit__(self, *exc):
        lib().orc_set_mutation(0)


# ---- single operations ------------------------------------------------------

def bf16_value(bits: int) -> float:
    return lib().orc_bf16_value(int(bits))


def fp16_value(bits: int) -> float:
    return lib().orc_fp16_value(int(bits))


def bf16_round(x: float) -> int:
    return lib().orc_bf16_round(float(x))


def rmsnorm(x, w_bits: np.ndarray, eps: float) -> np.ndarray:
    x = _f64(x)
    w = np.ascontiguousarray(w_bits, dtype=np.uint16)
    out = np.empty_like(x)
    lib().orc_rmsnorm(_p(x), _p(w), x.size, eps, _p(out))
    return out


def gemv_bf16(W_bits: np.ndarray, x) -> np.ndarray:
    W = np.ascontiguousarray(W_bits, dtype=np.uint16)
    x = _f64(x)
    N, K = W.shape
    y = np.empty(N, dtype=np.float64)
    lib().orc_gemv_bf16(_p(W), N, K, _p(x), _p(y))
    return y


def rope(h, pos: int, theta: float, interleaved: bool = False) -> np.ndarray:
    """h: [n_heads, d] -> rotated copy (rotate-half pairs, or interleaved pairs)."""
    h = _f64(h).copy()
    n, d = h.shape
    fn = lib().orc_rope_interleaved if interleaved else lib().orc_rope
    fn(_p(h), n, d, pos, theta)
    return h


def attention_head(q, K_bits: np.ndarray, V_bits: np.ndarray) -> np.ndarray:
    """q: [d]; K, V: bf16 bits [n][d] of one KV head."""
    q = _f64(q)
    K = np.ascontiguousarray(K_bits, dtype=np.uint16)
    V = np.ascontiguousarray(V_bits, dtype=np.uint16)
    n, d = K.shape
    o = np.empty(d, dtype=np.float64)
    lib().orc_attention_head(_p(q), _p(K), _p(V), n, d, _p(o))
    return o


def kv_head_of(h: int, n_q: int, n_kv: int) -> int:
    return lib().orc_kv_head_of(h, n_q, n_kv)


def silu(z: float) -> float:
    return lib().orc_silu(float(z))


def swiglu(g, u) -> np.ndarray:
    g, u = _f64(g), _f64(u)
    a = np.empty_like(g)
    lib().orc_swiglu(_p(g), _p(u), g.size, _p(a))
    return a


def quantize_act(z) -> tuple[np.ndarray, np.ndarray]:
    z = _f64(z)
    q = np.empty(z.size, dtype=np.int8)
    d = np.empty(z.size // 32, dtype=np.float32)
    lib().orc_quantize_act(_p(z), z.size, _p(q), _p(d))
    return q, d


def q4_blockdots(packed: np.ndarray, qx: np.ndarray) -> np.ndarray:
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    qx = np.ascontiguousarray(qx, dtype=np.int8)
    N = packed.shape[0]
    K = packed.shape[1] * 2
    out = np.empty((N, K // 32), dtype=np.int64)
    lib().orc_q4_blockdots(_p(packed), N, K, _p(qx), _p(out))
    return out


def gemv_q4(packed: np.ndarray, scales: np.ndarray, qx: np.ndarray, dx: np.ndarray) -> np.ndarray:
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint16)
    qx = np.ascontiguousarray(qx, dtype=np.int8)
    dx = np.ascontiguousarray(dx, dtype=np.float32)
    N = packed.shape[0]
    K = packed.shape[1] * 2
    y = np.empty(N, dtype=np.float64)
    lib().orc_gemv_q4(_p(packed), _p(scales), N, K, _p(qx), _p(dx), _p(y))
    return y


def lm_head(x, norm_w_bits: np.ndarray, W_bits: np.ndarray, eps: float = 1e-6):
    """Final RMSNorm x weight, logits = W n (W bf16 bits [V][H]), and the greedy
    token (the lowest index of the largest logit).  Returns (token, logits)."""
    x = _f64(x)
    nw = np.ascontiguousarray(norm_w_bits, dtype=np.uint16)
    W = np.ascontiguousarray(W_bits, dtype=np.uint16)
    V, H = W.shape
    logits = np.empty(V, dtype=np.float64)
    tok = lib().orc_lm_head(_p(x), H, _p(nw), _p(W), V, eps, _p(logits))
    return int(tok), logits


# ---- the stack ----------------------------------------------------------------

class OracleStack:
    """A decoder stack with its own bf16 KV cache, stepped one token at a time.

    layers: list of dicts with keys 'attn_norm', 'ffn_norm' (bf16 bits [H]) and
    either 'w' (list of 7 bf16 [out][in] arrays: q k v o gate up down) or
    'q4' (list of 7 (packed, scales) pairs).
    """

    def __init__(self, *, hidden, n_q_heads, n_kv_heads, head_dim, ffn, max_ctx, layers,
                 rms_eps=1e-6, rope_theta=1e4, q4=False, rope_interleaved=False):
        self.dims = Dims(hidden, n_q_heads, n_kv_heads, head_dim, ffn, max_ctx, int(q4),
                         int(rope_interleaved), rms_eps, rope_theta)
        self.n_layers = len(layers)
        self.hidden = hidden
        self.kv_len = 0
        self._keep = []
        self.kcache = np.zeros((self.n_layers, n_kv_heads, max_ctx, head_dim), dtype=np.uint16)
        self.vcache = np.zeros_like(self.kcache)
        self._layers = (Layer * self.n_layers)()
        for i, lw in enumerate(layers):
            L = self._layers[i]
            an = np.ascontiguousarray(lw["attn_norm"], dtype=np.uint16)
            fn = np.ascontiguousarray(lw["ffn_norm"], dtype=np.uint16)
            self._keep += [an, fn]
            L.attn_norm, L.ffn_norm = _p(an), _p(fn)
            for s in range(7):
                if q4:
                    pk, sc = lw["q4"][s]
                    pk = np.ascontiguousarray(pk, dtype=np.uint8)
                    sc = np.ascontiguousarray(sc, dtype=np.uint16)
                    self._keep += [pk, sc]
                    L.q[s], L.s[s] = _p(pk), _p(sc)
                else:
                    w = np.ascontiguousarray(lw["w"][s], dtype=np.uint16)
                    self._keep.append(w)
                    L.w[s] = _p(w)
            L.kcache = _p(self.kcache[i])
            L.vcache = _p(self.vcache[i])

    def load_kv(self, layer: int, k_bits: np.ndarray, v_bits: np.ndarray):
        """Prefilled rows [n_kv][n_pos][d] (already rotated k, raw v)."""
        n = k_bits.shape[1]
        self.kcache[layer, :, :n, :] = k_bits
        self.vcache[layer, :, :n, :] = v_bits
        self.kv_len = n

    def step(self, x, pos: int, per_layer: bool = False):
        """One token: returns the last layer's output (and every layer's if asked)."""
        assert pos == self.kv_len, "decode is strictly sequential"
        x = _f64(x)
        out = np.empty(self.hidden, dtype=np.float64)
        taps = np.empty((self.n_layers, self.hidden), dtype=np.float64) if per_layer else None
        rc = lib().orc_stack_step(ctypes.byref(self.dims), self._layers, self.n_layers, pos,
                                  _p(x), _p(out), _p(taps))
        if rc != 0:
            raise ValueError(f"oracle step failed (rc={rc}) at pos {pos}")
        self.kv_len = pos + 1
        return (out, taps) if per_layer else out

    def layer_step(self, layer: int, x, pos: int, qtap: bool = False, qgiven=None,
                   zout: bool = False, kv_given: bool = False, kvz: bool = False):
        """One layer alone (does not advance kv_len).

        For q4 stacks: qtap returns, with the output, the int8 codes and scales
        of the four GEMV inputs (n1, o, n2, a) as a list of (codes, scales)
        pairs, or (codes, scales, z) triples with zout, z being the fp64 vector
        each slot quantizes.  qgiven: four entries, each a (codes, scales) pair
        the layer uses for that GEMV input instead of quantizing it, or None to
        quantize it here.  Any stack: kv_given leaves the cache row pos as it
        is (the caller wrote this token's k, v there) instead of appending;
        kvz also returns this token's rotated k and v in fp64 ([n_kv][d] each),
        before the storage rounding.  Returns out, (out, codes), (out, kv) or
        (out, codes, kv) accordingly."""
        x = _f64(x)
        out = np.empty(self.hidden, dtype=np.float64)
        tap = QTap()
        arrays = None
        if qtap or zout or qgiven is not None:
            H, F = self.hidden, self.dims.ffn
            qd = self.dims.n_q_heads * self.dims.head_dim
            arrays = []
            for i, K in enumerate((H, qd, H, F)):
                g = qgiven[i] if qgiven is not None else None
                if g is not None:
                    qq = np.ascontiguousarray(g[0], np.int8)
                    dd = np.ascontiguousarray(g[1], np.float32)
                    tap.given |= 1 << i
                else:
                    qq, dd = np.empty(K, np.int8), np.empty(K // 32, np.float32)
                zz = np.empty(K, np.float64) if zout else None
                tap.q[i], tap.d[i], tap.z[i] = _p(qq), _p(dd), _p(zz)
                arrays.append((qq, dd, zz) if zout else (qq, dd))
        kv = None
        if kvz:
            nkv, d = self.dims.n_kv_heads, self.dims.head_dim
            kv = (np.empty((nkv, d), np.float64), np.empty((nkv, d), np.float64))
            tap.kz, tap.vz = _p(kv[0]), _p(kv[1])
        tap.kv_given = int(bool(kv_given))
        rc = lib().orc_layer_step(ctypes.byref(self.dims), ctypes.byref(self._layers[layer]), pos,
                                  _p(x), _p(out), ctypes.byref(tap))
        if rc != 0:
            raise ValueError(f"oracle layer step failed (rc={rc})")
        res = (out,)
        if qtap or zout:
            res += (arrays,)
        if kvz:
            res += (kv,)
        return res[0] if len(res) == 1 else res
