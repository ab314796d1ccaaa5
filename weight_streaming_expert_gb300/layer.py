"""Python face of the C ABI: ``MoELayer`` wraps one ``moe_layer_t`` handle.

PyTorch is used for device memory and streams only; tensors are passed to
the library as raw device pointers.
"""
from __future__ import annotations

import ctypes

import torch

from . import native as N


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_ptr(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


class MoELayer:
    """One routed-MoE layer (router + top-k + SwiGLU experts + combine).

    Weights (bf16, on the current CUDA device) are copied into the library at
    construction; the caller's tensors may be freed afterwards.
      w_router  [E, H]     w_gate_up [E, 2I, H] (gate rows first)   w_down [E, H, I]
    """

    def __init__(self, w_router, w_gate_up, w_down, topk: int, shared_gate_up=None, shared_down=None,
                 routed_scale: float = 1.0, bias_selection_only: bool = False):
        E, H = w_router.shape
        I = w_down.shape[2]
        for t in (w_router, w_gate_up, w_down):
            if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
                raise ValueError("weights must be contiguous bf16 CUDA tensors")
        if tuple(w_gate_up.shape) != (E, 2 * I, H) or tuple(w_down.shape) != (E, H, I):
            raise ValueError("weight shapes must be [E,H], [E,2I,H], [E,H,I]")
        if (shared_gate_up is None) != (shared_down is None):
            raise ValueError("give both shared_gate_up and shared_down, or neither")
        if shared_gate_up is not None and (tuple(shared_gate_up.shape) != (2 * I, H)
                                           or tuple(shared_down.shape) != (H, I)):
            raise ValueError("shared expert shapes must be [2I,H] and [H,I]")
        self.hidden, self.n_experts, self.topk, self.inter = H, E, topk, I
        self.shared = shared_gate_up is not None
        self.device = w_router.device
        L = N.lib()
        opts = N.moe_layer_opts_t(None if shared_gate_up is None else shared_gate_up.data_ptr(),
                                  None if shared_down is None else shared_down.data_ptr(),
                                  float(routed_scale), 1 if bias_selection_only else 0)
        with torch.cuda.device(self.device):
            h = L.moe_create_ex(H, E, topk, I, _ptr(w_router), _ptr(w_gate_up), _ptr(w_down), ctypes.byref(opts))
        if not h:
            raise N.MoEError("moe_create", N.MOE_ERR_INVALID_ARG, N.last_error())
        self._h = ctypes.c_void_p(h)

    @classmethod
    def fp8(cls, w_router, q_gate_up, s_gate_up, q_down, s_down, topk: int):
        """A layer with fp8 (E4M3) expert weights and fp32 per-row scales
        (``moe_create_fp8``): w_router bf16 [E,H]; q_gate_up uint8 [E,2I,H],
        s_gate_up fp32 [E,2I]; q_down uint8 [E,H,I], s_down fp32 [E,H]."""
        E, H = w_router.shape
        I = q_down.shape[2]
        if w_router.dtype != torch.bfloat16 or q_gate_up.dtype != torch.uint8 or q_down.dtype != torch.uint8:
            raise ValueError("w_router must be bf16 and the codes uint8")
        if s_gate_up.dtype != torch.float32 or s_down.dtype != torch.float32:
            raise ValueError("the row scales must be fp32")
        for t in (w_router, q_gate_up, s_gate_up, q_down, s_down):
            if not t.is_cuda or not t.is_contiguous():
                raise ValueError("weights must be contiguous CUDA tensors")
        if (tuple(q_gate_up.shape) != (E, 2 * I, H) or tuple(q_down.shape) != (E, H, I)
                or tuple(s_gate_up.shape) != (E, 2 * I) or tuple(s_down.shape) != (E, H)):
            raise ValueError("shapes must be [E,2I,H], [E,2I], [E,H,I], [E,H]")
        self = cls.__new__(cls)
        self.hidden, self.n_experts, self.topk, self.inter = H, E, topk, I
        self.shared = False
        self.device = w_router.device
        with torch.cuda.device(self.device):
            h = N.lib().moe_create_fp8(H, E, topk, I, _ptr(w_router), _ptr(q_gate_up), _ptr(s_gate_up),
                                       _ptr(q_down), _ptr(s_down))
        if not h:
            raise N.MoEError("moe_create_fp8", N.MOE_ERR_INVALID_ARG, N.last_error())
        self._h = ctypes.c_void_p(h)
        return self

    @property
    def handle(self):
        return self._h

    def info(self) -> N.moe_info_t:
        o = N.moe_info_t()
        N.check("moe_get_info", N.lib().moe_get_info(self._h, ctypes.byref(o)))
        return o

    def set_router_bias(self, bias):
        """bias: fp32 [E] tensor (any device) or None."""
        if bias is not None:
            bias = bias.to(device=self.device, dtype=torch.float32).contiguous()
        N.check("moe_set_router_bias", N.lib().moe_set_router_bias(self._h, _ptr(bias)))
        torch.cuda.synchronize(self.device)

    def forward(self, x, out=None, topk_idx=None, topk_w=None, stream=None, pdl=True, graph=False,
                trace=False, out_f32=False, test_skip_arrival=False):
        """x: bf16 [M, H] CUDA.  Returns (out [M,H], topk_idx [M,k] int32):
        out is bf16, or with out_f32 the fp32 combine before its rounding (the
        partial output of one slice of a tensor-parallel split)."""
        M = x.shape[0]
        if x.dtype != torch.bfloat16 or not x.is_contiguous() or x.shape[1] != self.hidden:
            raise ValueError("x must be contiguous bf16 [M, hidden]")
        if out is None:
            out = torch.empty((M, self.hidden), dtype=torch.float32 if out_f32 else torch.bfloat16,
                              device=x.device)
        elif out.dtype != (torch.float32 if out_f32 else torch.bfloat16) or not out.is_contiguous():
            raise ValueError("out must be contiguous " + ("fp32" if out_f32 else "bf16"))
        if topk_idx is None:
            topk_idx = torch.empty((M, self.topk), dtype=torch.int32, device=x.device)
        flags = ((0 if pdl else N.MOE_FWD_NO_PDL) | (N.MOE_FWD_GRAPH if graph else 0)
                 | (N.MOE_FWD_TRACE if trace else 0) | (N.MOE_FWD_OUT_F32 if out_f32 else 0)
                 | (N.MOE_FWD_TEST_SKIP_ARRIVAL if test_skip_arrival else 0))
        rc = N.lib().moe_forward_ex(self._h, _ptr(x), _ptr(out), _ptr(topk_idx), _ptr(topk_w), M,
                                    _stream_ptr(stream), flags)
        N.check("moe_forward_ex", rc)
        return out, topk_idx

    __call__ = forward

    def forward_timed(self, x, out, topk_idx, events, stream=None):
        """Profiling launch: events = 2 torch.cuda.Event(enable_timing=True)."""
        st = stream if stream is not None else torch.cuda.current_stream()
        for e in events:
            if not e.cuda_event:      # torch creates the CUDA event on first record
                e.record(st)
        arr = (ctypes.c_void_p * 2)(*[ctypes.c_void_p(e.cuda_event) for e in events[:2]])
        rc = N.lib().moe_forward_timed(self._h, _ptr(x), _ptr(out), _ptr(topk_idx), x.shape[0],
                                       _stream_ptr(stream), arr)
        N.check("moe_forward_timed", rc)

    def set_grid(self, ctas: int = 0):
        """CTAs of every later forward call (0: one per SM).  Synchronises."""
        N.check("moe_set_grid", N.lib().moe_set_grid(self._h, int(ctas)))

    def set_wait_limit(self, ns: int = 0):
        """Limit of the kernel's bounded waits in ns (0: the default)."""
        N.check("moe_set_wait_limit", N.lib().moe_set_wait_limit(self._h, int(ns)))

    def read_trace(self):
        """Phase timestamps of the last traced call: int64 numpy [SMs, 16] (ns;
        slot 11 is the CTA's gate/up tile count).  Synchronises."""
        import numpy as np
        n = self.info().n_sms * N.TRACE_SLOTS
        buf = np.zeros(n, np.uint64)
        rc = N.lib().moe_read_trace(self._h, buf.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64)), n)
        if rc < 0:
            N.check("moe_read_trace", -rc)
        return buf.astype(np.int64).reshape(-1, N.TRACE_SLOTS)

    def status(self) -> int:
        """Synchronises; returns the sticky device status (0 = ok) and clears it."""
        return N.lib().moe_get_status(self._h)

    def read_routing(self, M: int):
        """Last call's on-device compaction as numpy arrays (synchronises)."""
        import numpy as np
        np_ = M * (self.topk + (1 if self.shared else 0))  # pairs, the shared expert's last
        cap = max(1, np_)
        ng, na = ctypes.c_int(), ctypes.c_int()
        ge = np.zeros(cap, np.int32)
        gs = np.zeros(cap, np.int32)
        gc = np.zeros(cap, np.int32)
        pl = np.zeros(cap, np.int32)
        pw = np.zeros(cap, np.float32)
        i32 = ctypes.POINTER(ctypes.c_int32)
        rc = N.lib().moe_read_routing(self._h, M, ctypes.byref(ng), ctypes.byref(na),
                                      ge.ctypes.data_as(i32), gs.ctypes.data_as(i32), gc.ctypes.data_as(i32),
                                      pl.ctypes.data_as(i32),
                                      pw.ctypes.data_as(ctypes.POINTER(ctypes.c_float)), cap)
        N.check("moe_read_routing", rc)
        n = ng.value
        return dict(n_groups=n, n_active=na.value, grp_expert=ge[:n], grp_start=gs[:n], grp_cnt=gc[:n],
                    pair_list=pl[:np_], pair_w=pw[:np_])

    def close(self):
        if getattr(self, "_h", None):
            N.lib().moe_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def tp_slice(w_gate_up, w_down, rank: int, world: int):
    """The expert weights one GPU of a ``world``-way tensor-parallel split
    holds (the post's TP4): gate rows and up rows [rank*I/G, (rank+1)*I/G)
    of every expert and the matching down columns, as contiguous tensors
    ``(w_gate_up [E, 2I/G, H], w_down [E, H, I/G])`` on the weights' device.
    The router is not split: every GPU routes all tokens."""
    E, I2, H = w_gate_up.shape
    I = I2 // 2
    if I2 != 2 * I or tuple(w_down.shape) != (E, H, I) or world < 1 or I % world or not 0 <= rank < world:
        raise ValueError("need w_gate_up [E,2I,H], w_down [E,H,I] and I divisible by world")
    s = I // world
    lo, hi = rank * s, (rank + 1) * s
    gu = torch.cat([w_gate_up[:, lo:hi], w_gate_up[:, I + lo:I + hi]], dim=1).contiguous()
    return gu, w_down[:, :, lo:hi].contiguous()


def combine_partials(parts, out=None, stream=None):
    """bf16( parts[0] + parts[1] + ... ) in that order, one rounding
    (``moe_combine_partials``).  parts: fp32 CUDA tensor [G, M, H] (as an
    all-gather leaves the slices' fp32 outputs).  Returns bf16 [M, H]."""
    if parts.dtype != torch.float32 or not parts.is_cuda or not parts.is_contiguous() or parts.dim() != 3:
        raise ValueError("parts must be a contiguous fp32 CUDA tensor [G, M, H]")
    G, M, H = parts.shape
    if out is None:
        out = torch.empty((M, H), dtype=torch.bfloat16, device=parts.device)
    N.check("moe_combine_partials", N.lib().moe_combine_partials(_ptr(parts), G, M * H, _ptr(out),
                                                                 _stream_ptr(stream)))
    return out


class LmHead:
    """The bf16 vocabulary projection (``include/lm_head.h``): fp32 logits
    [M, V] = x [M, H] @ W [V, H]^T for M <= 16.  W (bf16, contiguous, on the
    current CUDA device) is copied into the library at construction."""

    def __init__(self, w):
        if w.dtype != torch.bfloat16 or not w.is_cuda or not w.is_contiguous() or w.dim() != 2:
            raise ValueError("w must be a contiguous bf16 CUDA tensor [vocab, hidden]")
        self.vocab, self.hidden = w.shape
        self.device = w.device
        with torch.cuda.device(self.device):
            h = N.lib().moe_lm_head_create(self.hidden, self.vocab, _ptr(w))
        if not h:
            raise N.MoEError("moe_lm_head_create", N.MOE_ERR_INVALID_ARG, N.last_error())
        self._h = ctypes.c_void_p(h)

    def __call__(self, x, logits=None, stream=None):
        return self.forward(x, logits, stream)

    def forward(self, x, logits=None, stream=None):
        """x: bf16 [M, H] CUDA.  Returns fp32 logits [M, V]."""
        if x.dtype != torch.bfloat16 or not x.is_contiguous() or x.shape[1] != self.hidden:
            raise ValueError("x must be contiguous bf16 [M, hidden]")
        if logits is None:
            logits = torch.empty((x.shape[0], self.vocab), dtype=torch.float32, device=x.device)
        rc = N.lib().moe_lm_head_forward(self._h, _ptr(x), _ptr(logits), x.shape[0], _stream_ptr(stream))
        N.check("moe_lm_head_forward", rc)
        return logits

    def status(self) -> int:
        return N.lib().moe_lm_head_get_status(self._h)

    def close(self):
        if getattr(self, "_h", None):
            N.lib().moe_lm_head_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
