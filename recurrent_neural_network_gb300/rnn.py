"""Thin ctypes binding of librnn (include/rnn.h): argument marshalling only.

Every step of the forward, backward-through-time and weight-gradient passes
runs in the library's CUDA kernels; this module passes device pointers
(``tensor.data_ptr()``), sizes and the current CUDA stream.  PyTorch is used
by callers for device memory and streams only.  There is no fallback: if the
library or a GPU is missing, the calls raise.
"""
from __future__ import annotations

import ctypes
import os

from . import synth

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "librnn.so")

RNN_OK = 0
ERRORS = {-1: "INVALID_ARG", -2: "UNSUPPORTED", -3: "LAUNCH", -4: "CUDA", -5: "TIMEOUT", -6: "NOMEM"}
FLAG_NO_WAVEFRONT = 0x1
FLAG_FORCE_STREAMING = 0x2
FLAG_FORCE_PERSISTENT = 0x4
FLAG_PROFILE = 0x8
FLAG_NO_PAIR = 0x20
FLAG_NO_GRAPH = 0x40
FLAG_NO_PDL = 0x80
FLAG_TEST_SKIP_PUBLISH = 0x100
FLAG_NO_TRANSPOSED = 0x200
FLAG_FORCE_TRANSPOSED = 0x400
FLAG_NO_FUSED_POINT = 0x800
FLAG_NO_PERSIST_CLUSTER = 0x1000
FLAG_BIDIRECTIONAL = 0x2000
FLAG_FP8_STASH = 0x4000
FLAG_PERSIST_CLUSTER_SYNC = 0x8000
FLAG_NO_STACK = 0x10000
FLAG_FORCE_STACK = 0x20000
FLAG_NO_STACK_BWD = 0x40000
FLAG_SLIM_STEP = 0x80000
FLAG_STEP_CHUNKS = 0x100000

# every symbol include/rnn.h declares
SYMBOLS = ["rnn_create", "rnn_destroy", "rnn_get_sizes", "rnn_pack_weights", "rnn_fwd", "rnn_bwd_data",
           "rnn_bwd_weights", "rnn_sync_status", "rnn_strerror", "rnn_describe", "rnn_launch_count",
           "rnn_profile_query", "rnn_gemm_bf16", "rnn_bias_grad_static", "rnn_set_lengths",
           "rnn_quantize_e4m3_rows"]
BIAS_STATIC_FLOATS = 1 << 20


class RnnError(RuntimeError):
    def __init__(self, code, what):
        super().__init__(f"{what}: {ERRORS.get(code, code)} ({code})")
        self.code = code


class Desc(ctypes.Structure):
    _fields_ = [("cell", ctypes.c_int), ("layers", ctypes.c_int), ("T", ctypes.c_int), ("B", ctypes.c_int),
                ("input", ctypes.c_int), ("hidden", ctypes.c_int), ("mode", ctypes.c_int),
                ("flags", ctypes.c_uint), ("timeout_ns", ctypes.c_longlong), ("chunk", ctypes.c_int)]


_lib = None


def load(path: str = LIB_PATH):
    """Load librnn.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"librnn.so is missing at {path}; build it with "
                           "`python -m recurrent_neural_network_gb300.build`")
    lib = ctypes.CDLL(path)
    vp, sz, ci = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
    H = ctypes.c_void_p  # handle
    lib.rnn_create.argtypes = [ctypes.POINTER(Desc), ctypes.POINTER(H)]
    lib.rnn_destroy.argtypes = [H]
    lib.rnn_get_sizes.argtypes = [H] + [ctypes.POINTER(sz)] * 4
    lib.rnn_pack_weights.argtypes = [H, vp, vp, vp]
    lib.rnn_fwd.argtypes = [H] + [vp] * 10
    lib.rnn_bwd_data.argtypes = [H] + [vp] * 12
    lib.rnn_bwd_weights.argtypes = [H, vp, vp, vp, vp, ci, vp, vp]
    lib.rnn_sync_status.argtypes = [H, vp, vp]
    lib.rnn_strerror.argtypes = [ci]
    lib.rnn_strerror.restype = ctypes.c_char_p
    lib.rnn_describe.argtypes = [H, ctypes.c_char_p, sz]
    lib.rnn_launch_count.restype = ctypes.c_ulonglong
    lib.rnn_profile_query.argtypes = [H, ci, ctypes.c_char_p, ctypes.POINTER(ci), ctypes.POINTER(ctypes.c_ulonglong),
                                      ctypes.POINTER(ctypes.c_double), ci]
    lib.rnn_gemm_bf16.argtypes = [ci, ci, ci, vp, ctypes.c_longlong, ci, vp, ctypes.c_longlong, ci, vp,
                                  ctypes.c_longlong, vp, ci, vp]
    lib.rnn_bias_grad_static.argtypes = [H, vp, vp, ci, vp]
    lib.rnn_set_lengths.argtypes = [H, ctypes.POINTER(ci)]
    lib.rnn_quantize_e4m3_rows.argtypes = [ci, ci, vp, vp, vp, vp]
    for name in SYMBOLS:
        if name != "rnn_strerror" and name != "rnn_launch_count":
            getattr(lib, name).restype = ci
    _lib = lib
    return lib


def _ptr(t):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def check(rc, what):
    if rc != RNN_OK:
        raise RnnError(rc, what)


def launch_count() -> int:
    return int(load().rnn_launch_count())


def gemm_bf16(A, B, D, M, N, K, lda, ldb, ldd, a_mn=False, b_mn=False, bias=None, accumulate=False, stream=None):
    """D[m][n] = sum_k A(m,k) B(n,k) (+bias) (+D) on the tcgen05 engine (test hook)."""
    check(load().rnn_gemm_bf16(M, N, K, _ptr(A), lda, int(a_mn), _ptr(B), ldb, int(b_mn), _ptr(D), ldd, _ptr(bias),
                               int(accumulate), _stream(stream)), "rnn_gemm_bf16")


def quantize_e4m3_rows(w, q, scale, stream=None):
    """Per-row e4m3 quantisation of a bf16 [rows][cols] device tensor (test hook of the fp8 stash)."""
    rows, cols = w.shape
    check(load().rnn_quantize_e4m3_rows(rows, cols, _ptr(w), _ptr(q), _ptr(scale), _stream(stream)),
          "rnn_quantize_e4m3_rows")


class RNN:
    """One handle of librnn: a fixed (cell, layers, T, B, input, hidden, mode)."""

    def __init__(self, cell, layers, T, B, input, hidden, mode, flags=0, timeout_ns=0, chunk=0):
        self.lib = load()
        self.desc = Desc(cell, layers, T, B, input, hidden, mode, flags, timeout_ns, chunk)
        h = ctypes.c_void_p()
        check(self.lib.rnn_create(ctypes.byref(self.desc), ctypes.byref(h)), "rnn_create")
        self.h = h
        self.cell, self.layers, self.T, self.B, self.input, self.hidden, self.mode = \
            cell, layers, T, B, input, hidden, mode
        self.D = 2 if flags & FLAG_BIDIRECTIONAL else 1

    @classmethod
    def for_workload(cls, wl: synth.Workload, **kw):
        if wl.directions == 2:
            kw["flags"] = kw.get("flags", 0) | FLAG_BIDIRECTIONAL
        return cls(wl.cell, wl.layers, wl.T, wl.B, wl.input, wl.hidden, wl.mode, **kw)

    def close(self):
        if self.h:
            self.lib.rnn_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def sizes(self):
        s = [ctypes.c_size_t() for _ in range(4)]
        check(self.lib.rnn_get_sizes(self.h, *[ctypes.byref(v) for v in s]), "rnn_get_sizes")
        return dict(user_weights=s[0].value, packed_weights=s[1].value, reserve=s[2].value, workspace=s[3].value)

    def describe(self) -> str:
        buf = ctypes.create_string_buffer(512)
        check(self.lib.rnn_describe(self.h, buf, 512), "rnn_describe")
        return buf.value.decode()

    def pack_weights(self, w_user, w_packed, stream=None):
        check(self.lib.rnn_pack_weights(self.h, _ptr(w_user), _ptr(w_packed), _stream(stream)), "rnn_pack_weights")

    def fwd(self, x, w_packed, y, ws, h0=None, c0=None, hT=None, cT=None, reserve=None, stream=None):
        check(self.lib.rnn_fwd(self.h, _ptr(x), _ptr(h0), _ptr(c0), _ptr(w_packed), _ptr(y), _ptr(hT), _ptr(cT),
                               _ptr(reserve), _ptr(ws), _stream(stream)), "rnn_fwd")

    def bwd_data(self, dy, w_packed, reserve, ws, dhT=None, dcT=None, h0=None, c0=None, dx=None, dh0=None, dc0=None,
                 stream=None):
        check(self.lib.rnn_bwd_data(self.h, _ptr(dy), _ptr(dhT), _ptr(dcT), _ptr(w_packed), _ptr(h0), _ptr(c0),
                                    _ptr(dx), _ptr(dh0), _ptr(dc0), _ptr(reserve), _ptr(ws), _stream(stream)),
              "rnn_bwd_data")

    def bwd_weights(self, x, reserve, dw, ws, h0=None, accumulate=False, stream=None):
        check(self.lib.rnn_bwd_weights(self.h, _ptr(x), _ptr(h0), _ptr(reserve), _ptr(dw), int(accumulate), _ptr(ws),
                                       _stream(stream)), "rnn_bwd_weights")

    def set_lengths(self, lens=None):
        """Per-sequence lengths (non-increasing, 1..T) for later calls; None = all T."""
        if lens is None:
            check(self.lib.rnn_set_lengths(self.h, None), "rnn_set_lengths")
            return
        lens = [int(v) for v in lens]
        if len(lens) != self.B:
            raise ValueError(f"set_lengths: {len(lens)} lengths for a batch of {self.B}")
        arr = (ctypes.c_int * len(lens))(*lens)
        check(self.lib.rnn_set_lengths(self.h, arr), "rnn_set_lengths")

    def bias_grad_static(self, reserve, dw, accumulate=False, stream=None):
        """Bias gradients into dw using the library's fixed scratch array (no workspace)."""
        check(self.lib.rnn_bias_grad_static(self.h, _ptr(reserve), _ptr(dw), int(accumulate), _stream(stream)),
              "rnn_bias_grad_static")

    def sync_status(self, ws, stream=None) -> int:
        return int(self.lib.rnn_sync_status(self.h, _ptr(ws), _stream(stream)))

    def profile(self, reset=True):
        """{kernel class: (launches, total_ms)} of the calls since the last reset (needs FLAG_PROFILE)."""
        n = ctypes.c_int()
        check(self.lib.rnn_profile_query(self.h, -1, None, ctypes.byref(n), None, None, 0), "rnn_profile_query")
        out = {}
        for k in range(n.value):
            name = ctypes.create_string_buffer(32)
            cnt = ctypes.c_ulonglong()
            ms = ctypes.c_double()
            check(self.lib.rnn_profile_query(self.h, k, name, None, ctypes.byref(cnt), ctypes.byref(ms), 0),
                  "rnn_profile_query")
            out[name.value.decode()] = (int(cnt.value), float(ms.value))
        if reset:
            self.lib.rnn_profile_query(self.h, -1, None, None, None, None, 1)
        return out
