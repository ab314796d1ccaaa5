"""ctypes wrapper around the C++ CPU oracle (test infrastructure only).

bf16 tensors cross this boundary as numpy ``uint16`` arrays holding the bf16
bit patterns.  Every function here only marshals arguments; the arithmetic is
in ``moe_oracle.cpp``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.cpp")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

# -O2 without fast-math and without FMA contraction: the rounding sequence is
# exactly the one the source spells out, on x86-64 and aarch64 alike.
CXXFLAGS = ["-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(src: str = _SRC, out: str = _LIB_PATH, force: bool = False) -> str:
    """Compile the oracle into a shared library; returns its path."""
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["g++", *CXXFLAGS, src, "-o", tmp], check=True)
    os.replace(tmp, out)
    return out


def load(path: str | None = None):
    """Load (building first if needed) and declare the oracle's C symbols."""
    global _lib
    with _lock:
        if path is None and _lib is not None:
            return _lib
        p = path or build()
        lib = ctypes.CDLL(p)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        f32p = ctypes.POINTER(ctypes.c_float)
        i32p = ctypes.POINTER(ctypes.c_int32)
        ci = ctypes.c_int
        lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_f32.restype = ctypes.c_float
        lib.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
        lib.oracle_f32_to_bf16.restype = ctypes.c_uint16
        lib.oracle_swiglu_bf16.argtypes = [ctypes.c_float, ctypes.c_float]
        lib.oracle_swiglu_bf16.restype = ctypes.c_uint16
        lib.oracle_router_logits.argtypes = [ci, ci, ci, u16p, u16p, f32p, f32p]
        lib.oracle_topk_softmax.argtypes = [ci, ci, ci, f32p, i32p, f32p]
        lib.oracle_weights_for_set.argtypes = [ci, ci, f32p, i32p, f32p]
        lib.oracle_expert_swiglu.argtypes = [ci, ci, u16p, u16p, u16p]
        lib.oracle_expert_down.argtypes = [ci, ci, u16p, u16p, f32p]
        lib.oracle_moe_forward.argtypes = [ci, ci, ci, ci, ci, u16p, u16p, f32p, u16p, u16p,
                                           i32p, f32p, i32p, f32p, f32p, u16p, u16p]
        lib.oracle_lm_head.argtypes = [ci, ci, ci, u16p, u16p, f32p]
        u8p = ctypes.POINTER(ctypes.c_uint8)
        lib.oracle_e4m3_to_f32.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_to_f32.restype = ctypes.c_float
        lib.oracle_moe_forward_fp8.argtypes = [ci, ci, ci, ci, ci, u16p, u16p, f32p, u8p, f32p, u8p, f32p,
                                               i32p, f32p, i32p, f32p, f32p, u16p]
        lib.oracle_moe_forward_ex.argtypes = [ci, ci, ci, ci, ci, u16p, u16p, f32p, ci, u16p, u16p, u16p, u16p,
                                              ctypes.c_float, i32p, f32p, i32p, f32p, f32p, u16p, u16p]
        for name in ("oracle_router_logits", "oracle_topk_softmax", "oracle_weights_for_set",
                     "oracle_expert_swiglu", "oracle_expert_down", "oracle_moe_forward", "oracle_lm_head",
                     "oracle_moe_forward_ex", "oracle_moe_forward_fp8"):
            getattr(lib, name).restype = ci
        if path is None:
            _lib = lib
        return lib


def _p(a, ctype):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _u16(a):
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, f"bf16 arrays are passed as uint16 bits, got {a.dtype}"
    return a


class Oracle:
    """Bound oracle library (``path`` selects an alternative build)."""

    def __init__(self, path: str | None = None):
        self.lib = load(path)

    # scalar helpers -----------------------------------------------------
    def bf16_to_f32(self, b: int) -> float:
        return float(self.lib.oracle_bf16_to_f32(int(b)))

    def f32_to_bf16(self, f: float) -> int:
        return int(self.lib.oracle_f32_to_bf16(float(f)))

    def swiglu_bf16(self, g: float, u: float) -> int:
        return int(self.lib.oracle_swiglu_bf16(float(g), float(u)))

    # steps ------------------------------------------------------------------
    def router_logits(self, x, w_router, bias=None):
        x, w_router = _u16(x), _u16(w_router)
        M, H = x.shape
        E = w_router.shape[0]
        logits = np.zeros((M, E), np.float32)
        b = None if bias is None else np.ascontiguousarray(bias, np.float32)
        rc = self.lib.oracle_router_logits(M, H, E, _p(x, ctypes.c_uint16), _p(w_router, ctypes.c_uint16),
                                           _p(b, ctypes.c_float), _p(logits, ctypes.c_float))
        assert rc == 0
        return logits

    def lm_head(self, x, w):
        """fp32 logits [M, V] of bf16 tokens x [M, H] and projection w [V, H]."""
        x, w = _u16(x), _u16(w)
        M, H = x.shape
        V = w.shape[0]
        assert w.shape == (V, H)
        logits = np.zeros((M, V), np.float32)
        rc = self.lib.oracle_lm_head(M, H, V, _p(x, ctypes.c_uint16), _p(w, ctypes.c_uint16),
                                     _p(logits, ctypes.c_float))
        assert rc == 0
        return logits

    def topk_softmax(self, logits, k):
        logits = np.ascontiguousarray(logits, np.float32)
        M, E = logits.shape
        idx = np.zeros((M, k), np.int32)
        w = np.zeros((M, k), np.float32)
        rc = self.lib.oracle_topk_softmax(M, E, k, _p(logits, ctypes.c_float), _p(idx, ctypes.c_int32),
                                          _p(w, ctypes.c_float))
        assert rc == 0
        return idx, w

    def weights_for_set(self, logits_row, idx_row):
        logits_row = np.ascontiguousarray(logits_row, np.float32)
        idx_row = np.ascontiguousarray(idx_row, np.int32)
        w = np.zeros(idx_row.shape[0], np.float32)
        rc = self.lib.oracle_weights_for_set(logits_row.shape[0], idx_row.shape[0],
                                             _p(logits_row, ctypes.c_float), _p(idx_row, ctypes.c_int32),
                                             _p(w, ctypes.c_float))
        assert rc == 0
        return w

    def expert_swiglu(self, x_row, w_gate_up_e):
        x_row, w_gate_up_e = _u16(x_row), _u16(w_gate_up_e)
        H = x_row.shape[0]
        I = w_gate_up_e.shape[0] // 2
        h = np.zeros(I, np.uint16)
        rc = self.lib.oracle_expert_swiglu(H, I, _p(x_row, ctypes.c_uint16), _p(w_gate_up_e, ctypes.c_uint16),
                                           _p(h, ctypes.c_uint16))
        assert rc == 0
        return h

    def expert_down(self, h_row, w_down_e):
        h_row, w_down_e = _u16(h_row), _u16(w_down_e)
        I = h_row.shape[0]
        H = w_down_e.shape[0]
        y = np.zeros(H, np.float32)
        rc = self.lib.oracle_expert_down(H, I, _p(h_row, ctypes.c_uint16), _p(w_down_e, ctypes.c_uint16),
                                         _p(y, ctypes.c_float))
        assert rc == 0
        return y

    # whole layer ---------------------------------------------------------
    def moe_forward(self, x, w_router, w_gate_up, w_down, k, bias=None, idx_in=None, want_h=False,
                    shared_gate_up=None, shared_down=None, routed_scale=1.0, bias_selection_only=False):
        """Returns dict(out=u16[M,H], acc=f32[M,H], logits, idx, w, h?).  The
        layer variants: a shared expert (shared_gate_up [2I,H], shared_down
        [H,I]), a routed scaling factor, a bias for the selection only."""
        x, w_router, w_gate_up, w_down = _u16(x), _u16(w_router), _u16(w_gate_up), _u16(w_down)
        M, H = x.shape
        E = w_router.shape[0]
        I = w_down.shape[2]
        assert w_router.shape == (E, H)
        assert w_gate_up.shape == (E, 2 * I, H)
        assert w_down.shape == (E, H, I)
        sg = None if shared_gate_up is None else _u16(shared_gate_up)
        sd = None if shared_down is None else _u16(shared_down)
        if sg is not None:
            assert sg.shape == (2 * I, H) and sd is not None and sd.shape == (H, I)
        logits = np.zeros((M, E), np.float32)
        idx = np.zeros((M, k), np.int32)
        w = np.zeros((M, k), np.float32)
        acc = np.zeros((M, H), np.float32)
        out = np.zeros((M, H), np.uint16)
        h = np.zeros((M, k, I), np.uint16) if want_h else None
        b = None if bias is None else np.ascontiguousarray(bias, np.float32)
        ii = None if idx_in is None else np.ascontiguousarray(idx_in, np.int32)
        rc = self.lib.oracle_moe_forward_ex(
            M, H, E, k, I, _p(x, ctypes.c_uint16), _p(w_router, ctypes.c_uint16), _p(b, ctypes.c_float),
            1 if bias_selection_only else 0, _p(w_gate_up, ctypes.c_uint16), _p(w_down, ctypes.c_uint16),
            _p(sg, ctypes.c_uint16), _p(sd, ctypes.c_uint16), float(routed_scale), _p(ii, ctypes.c_int32),
            _p(logits, ctypes.c_float), _p(idx, ctypes.c_int32), _p(w, ctypes.c_float),
            _p(acc, ctypes.c_float), _p(h, ctypes.c_uint16), _p(out, ctypes.c_uint16))
        assert rc == 0, "oracle rejected its arguments"
        res = dict(out=out, acc=acc, logits=logits, idx=idx, w=w)
        if want_h:
            res["h"] = h
        return res

    # fp8 expert weights ---------------------------------------------------
    def e4m3_to_f32(self, code: int) -> float:
        return float(self.lib.oracle_e4m3_to_f32(int(code)))

    def moe_forward_fp8(self, x, w_router, q_gate_up, s_gate_up, q_down, s_down, k, bias=None, idx_in=None):
        """The layer with fp8 (E4M3) expert weights and per-row fp32 scales:
        q_gate_up u8 [E,2I,H], s_gate_up f32 [E,2I], q_down u8 [E,H,I],
        s_down f32 [E,H].  Returns dict(out, acc, logits, idx, w)."""
        x, w_router = _u16(x), _u16(w_router)
        q_gate_up = np.ascontiguousarray(q_gate_up, np.uint8)
        q_down = np.ascontiguousarray(q_down, np.uint8)
        s_gate_up = np.ascontiguousarray(s_gate_up, np.float32)
        s_down = np.ascontiguousarray(s_down, np.float32)
        M, H = x.shape
        E = w_router.shape[0]
        I = q_down.shape[2]
        assert q_gate_up.shape == (E, 2 * I, H) and s_gate_up.shape == (E, 2 * I)
        assert q_down.shape == (E, H, I) and s_down.shape == (E, H)
        logits = np.zeros((M, E), np.float32)
        idx = np.zeros((M, k), np.int32)
        w = np.zeros((M, k), np.float32)
        acc = np.zeros((M, H), np.float32)
        out = np.zeros((M, H), np.uint16)
        b = None if bias is None else np.ascontiguousarray(bias, np.float32)
        ii = None if idx_in is None else np.ascontiguousarray(idx_in, np.int32)
        rc = self.lib.oracle_moe_forward_fp8(
            M, H, E, k, I, _p(x, ctypes.c_uint16), _p(w_router, ctypes.c_uint16), _p(b, ctypes.c_float),
            _p(q_gate_up, ctypes.c_uint8), _p(s_gate_up, ctypes.c_float), _p(q_down, ctypes.c_uint8),
            _p(s_down, ctypes.c_float), _p(ii, ctypes.c_int32), _p(logits, ctypes.c_float),
            _p(idx, ctypes.c_int32), _p(w, ctypes.c_float), _p(acc, ctypes.c_float), _p(out, ctypes.c_uint16))
        assert rc == 0, "oracle rejected its arguments"
        return dict(out=out, acc=acc, logits=logits, idx=idx, w=w)
