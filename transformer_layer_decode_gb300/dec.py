"""ctypes binding of the decode library's C ABI (include/dec.h).

Argument marshalling only: every step of the decode runs in the library's
CUDA kernels.  PyTorch provides device memory and streams.  If the library has
not been built, :func:`load_library` raises; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libtld_gb300.so")
# the same library with the kernels' index checks compiled in (TLD_DEBUG_CHECKS)
DEBUG_LIB_PATH = os.path.join(_HERE, "_build", "libtld_gb300_debug.so")

# enum values of dec.h
DEC_OK, DEC_ERR_ARG, DEC_ERR_SHAPE, DEC_ERR_STATE = 0, -1, -2, -3
DEC_ERR_POS, DEC_ERR_CTX, DEC_ERR_CUDA, DEC_ERR_OOM, DEC_ERR_DEVICE = -4, -5, -6, -7, -8
DEC_W_BF16, DEC_W_Q4B32 = 0, 1
DEC_PLAN_FUSED, DEC_PLAN_UNFUSED, DEC_NO_GRAPH, DEC_NO_PDL, DEC_PLAN_PERSISTENT = 0, 1, 2, 4, 8
DEC_NO_L2_AHEAD, DEC_ATTN_GLOBAL_MERGE, DEC_PLAN_THREE, DEC_DEBUG_GUARDS = 16, 32, 64, 128
DEC_ROPE_INTERLEAVED, DEC_PAGED_KV, DEC_PLAN_FOUR, DEC_Q4_PUBLISH = 256, 512, 1024, 2048
DEC_FUSE_ATTN_OPROJ = 4096
DEC_T_ATTN_NORM, DEC_T_WQ, DEC_T_WK, DEC_T_WV, DEC_T_WO = 0, 1, 2, 3, 4
DEC_T_FFN_NORM, DEC_T_WGATE, DEC_T_WUP, DEC_T_WDOWN, DEC_T_SCALES = 5, 6, 7, 8, 16

# kernels of one layer, per plan
KERNEL_NAMES = ("norm_qkv_rope_append", "attention", "oproj_residual",
                "norm_gateup_swiglu", "down_residual")
KERNEL_NAMES_THREE = ("norm_qkv_rope_append", "attention_oproj_residual",
                      "norm_gateup_swiglu_down_residual")
KERNEL_NAMES_FOUR = ("norm_qkv_rope_append", "attention", "oproj_residual",
                     "norm_gateup_swiglu_down_residual")

EXPORTED = ("dec_create", "dec_load_weights", "dec_load_kv", "dec_read_kv", "dec_truncate_kv", "dec_step",
            "dec_load_lm_head", "dec_set_token_out", "dec_set_page_table",
            "dec_set_tap", "dec_set_dot_tap", "dec_set_timeline", "dec_sync_status",
            "dec_check_guards", "dec_get_info", "dec_launch_kernel",
            "dec_destroy", "dec_last_error", "dec_attention_noalloc")


class DecError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{msg} (code {code})")
        self.code = code


class ModelDesc(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("hidden", ctypes.c_int32),
                ("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("ffn", ctypes.c_int32),
                ("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_float),
                ("max_ctx", ctypes.c_int32), ("weight_fmt", ctypes.c_int32),
                ("flags", ctypes.c_int32)]


class Info(ctypes.Structure):
    _fields_ = [("kernels_per_layer", ctypes.c_int32), ("kernels_per_token", ctypes.c_int32),
                ("n_sm", ctypes.c_int32), ("kv_len", ctypes.c_int32),
                ("weight_bytes", ctypes.c_int64), ("kv_bytes", ctypes.c_int64),
                ("workspace_bytes", ctypes.c_int64), ("attn_grid", ctypes.c_int32),
                ("attn_cluster", ctypes.c_int32), ("page_rows", ctypes.c_int32),
                ("n_pages", ctypes.c_int32)]


_libs: dict = {}


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libtld_gb300.so (built by ``build.build()``), or the debug build of it
    (``DEBUG_LIB_PATH``, ``build.build(debug=True)``); raise if it is missing."""
    if path in _libs:
        return _libs[path]
    if not os.path.exists(path):
        raise RuntimeError(f"decode library not built: {path} is missing "
                           "(run transformer_layer_decode_gb300.build.build())")
    L = ctypes.CDLL(path)
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    sig = {
        "dec_create": [ctypes.POINTER(ModelDesc), ctypes.POINTER(vp)],
        "dec_load_weights": [vp, i32, i32, vp, sz],
        "dec_load_kv": [vp, i32, vp, vp, i32],
        "dec_read_kv": [vp, i32, vp, vp, i32, i32],
        "dec_load_lm_head": [vp, vp, vp, i32],
        "dec_set_token_out": [vp, vp, vp],
        "dec_set_page_table": [vp, vp, i32],
        "dec_truncate_kv": [vp, i32],
        "dec_step": [vp, vp, i32, vp, vp],
        "dec_set_tap": [vp, vp, vp, vp],
        "dec_set_timeline": [vp, vp],
        "dec_set_dot_tap": [vp, i32, i32, vp],
        "dec_sync_status": [vp, vp],
        "dec_check_guards": [vp],
        "dec_get_info": [vp, ctypes.POINTER(Info)],
        "dec_launch_kernel": [vp, i32, i32, i32, vp],
        "dec_destroy": [vp],
        "dec_attention_noalloc": [vp, vp, vp, i32, i32, i32, i32, i32, vp, vp],
    }
    for name, args in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = i32
    L.dec_last_error.argtypes = [vp]
    L.dec_last_error.restype = ctypes.c_char_p
    _libs[path] = L
    return L


def _ptr(x) -> int | None:
    """Address of a torch tensor, numpy array or raw int pointer (None passes NULL)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if isinstance(x, np.ndarray):
        assert x.flags.c_contiguous, "arrays must be C-contiguous"
        return x.ctypes.data
    if hasattr(x, "data_ptr"):
        assert x.is_contiguous(), "tensors must be contiguous"
        return x.data_ptr()
    raise TypeError(f"cannot take the address of {type(x)}")


def _nbytes(x) -> int:
    if isinstance(x, np.ndarray):
        return x.nbytes
    return x.numel() * x.element_size()


def _stream_handle(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def attention_noalloc(q, k_cache, v_cache, n_q_heads: int, n_kv_heads: int, head_dim: int,
                      ctx_stride: int, n: int, o, stream=None):
    """Decode attention through dec_attention_noalloc (no device allocation)."""
    L = load_library()
    rc = L.dec_attention_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), n_q_heads, n_kv_heads,
                                 head_dim, ctx_stride, n, _ptr(o), _stream_handle(stream))
    if rc != DEC_OK:
        raise DecError(rc, "dec_attention_noalloc rejected its arguments or failed to launch")


def noalloc_sync_status(stream=None):
    """Wait for `stream` and raise DecError if dec_attention_noalloc's kernel
    gave up a bounded wait on the current device (dec_sync_status(NULL, ...))."""
    L = load_library()
    rc = L.dec_sync_status(None, _stream_handle(stream))
    if rc != DEC_OK:
        raise DecError(rc, L.dec_last_error(None).decode())


@dataclass
class Shape:
    n_layers: int
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    max_ctx: int
    rms_eps: float = 1e-6
    rope_theta: float = 1e4
    weight_fmt: int = DEC_W_BF16


class Decoder:
    """One decode handle: weights, KV cache and the captured step graph."""

    def __init__(self, shape: Shape, *, unfused: bool = False, graph: bool = True,
                 pdl: bool = True, persistent: bool = False, l2_ahead: bool = True,
                 cluster_attn: bool = True, three: bool = False, four: bool = False,
                 guards: bool = False,
                 rope_interleaved: bool = False, paged_kv: bool = False,
                 q4_publish: bool = False, attn_oproj: bool = False,
                 lib_path: str | None = None):
        self.lib = load_library(lib_path or LIB_PATH)
        self.shape = shape
        flags = ((DEC_PLAN_UNFUSED if unfused else 0) | (0 if graph else DEC_NO_GRAPH)
                 | (0 if pdl else DEC_NO_PDL) | (DEC_PLAN_PERSISTENT if persistent else 0)
                 | (0 if l2_ahead else DEC_NO_L2_AHEAD)
                 | (0 if cluster_attn else DEC_ATTN_GLOBAL_MERGE)
                 | (DEC_PLAN_THREE if three else 0) | (DEC_PLAN_FOUR if four else 0)
                 | (DEC_DEBUG_GUARDS if guards else 0)
                 | (DEC_ROPE_INTERLEAVED if rope_interleaved else 0)
                 | (DEC_PAGED_KV if paged_kv else 0)
                 | (DEC_Q4_PUBLISH if q4_publish else 0)
                 | (DEC_FUSE_ATTN_OPROJ if attn_oproj else 0))
        self.desc = ModelDesc(shape.n_layers, shape.hidden, shape.n_q_heads, shape.n_kv_heads,
                              shape.head_dim, shape.ffn, shape.rms_eps, shape.rope_theta,
                              shape.max_ctx, shape.weight_fmt, flags)
        h = ctypes.c_void_p()
        rc = self.lib.dec_create(ctypes.byref(self.desc), ctypes.byref(h))
        if rc != DEC_OK:
            raise DecError(rc, self.lib.dec_last_error(None).decode())
        self.h = h

    def _check(self, rc: int):
        if rc != DEC_OK:
            raise DecError(rc, self.lib.dec_last_error(self.h).decode())

    def load_weights(self, layer: int, tensor: int, src):
        self._check(self.lib.dec_load_weights(self.h, layer, tensor, _ptr(src), _nbytes(src)))

    def load_kv(self, layer: int, k, v, n_pos: int | None = None):
        n = k.shape[1] if n_pos is None else n_pos
        self._check(self.lib.dec_load_kv(self.h, layer, _ptr(k), _ptr(v), n))

    def load_lm_head(self, final_norm, w):
        """final_norm: bf16 bits [hidden]; w: bf16 bits [vocab][hidden] (host or device)."""
        self._check(self.lib.dec_load_lm_head(self.h, _ptr(final_norm), _ptr(w), w.shape[0]))

    def set_token_out(self, token_out=None, logits=None):
        self._check(self.lib.dec_set_token_out(self.h, _ptr(token_out), _ptr(logits)))

    def set_page_table(self, pages):
        pages = np.ascontiguousarray(pages, dtype=np.int32)
        self._check(self.lib.dec_set_page_table(self.h, _ptr(pages), pages.size))

    def read_kv(self, layer: int, first_pos: int, n_pos: int):
        """Rows [first_pos, first_pos + n_pos) of one layer's cache: (K, V) bf16
        bits [n_kv_heads][n_pos][head_dim] as numpy uint16."""
        sh = (self.shape.n_kv_heads, n_pos, self.shape.head_dim)
        k, v = np.empty(sh, np.uint16), np.empty(sh, np.uint16)
        self._check(self.lib.dec_read_kv(self.h, layer, _ptr(k), _ptr(v), first_pos, n_pos))
        return k, v

    def truncate_kv(self, n_pos: int):
        self._check(self.lib.dec_truncate_kv(self.h, n_pos))

    def step(self, emb, pos: int, out, stream=None):
        self._check(self.lib.dec_step(self.h, _ptr(emb), pos, _ptr(out), _stream_handle(stream)))

    def set_tap(self, per_layer_out=None, qact=None, qscale=None):
        self._check(self.lib.dec_set_tap(self.h, _ptr(per_layer_out), _ptr(qact), _ptr(qscale)))

    def set_dot_tap(self, layer: int = 0, kernel: int = 0, dots=None):
        self._check(self.lib.dec_set_dot_tap(self.h, layer, kernel, _ptr(dots)))

    def set_timeline(self, buf=None):
        self._check(self.lib.dec_set_timeline(self.h, _ptr(buf)))

    def sync_status(self, stream=None):
        self._check(self.lib.dec_sync_status(self.h, _stream_handle(stream)))

    def check_guards(self):
        self._check(self.lib.dec_check_guards(self.h))

    def info(self) -> Info:
        inf = Info()
        self._check(self.lib.dec_get_info(self.h, ctypes.byref(inf)))
        return inf

    def launch_kernel(self, kernel: int, first_layer: int, count: int, stream=None):
        self._check(self.lib.dec_launch_kernel(self.h, kernel, first_layer, count,
                                               _stream_handle(stream)))

    def close(self):
        if getattr(self, "h", None):
            self.lib.dec_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
