"""Python binding of libmoegmm (the GB300 fused grouped expert MLP).

Argument marshalling only: every step of the layer runs in the library's CUDA kernels. The
functions below carry the C ABI's names (include/moegmm.h) and accept torch tensors (their
device pointers are passed) or raw integer addresses. `MoELayer` is plumbing on top: it
allocates the caller-owned buffers with torch and calls the same entry points.

There is no fallback: if the shared library is missing, `load()` raises.
"""
from __future__ import annotations

import ctypes
import math
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libmoegmm.so")

PREC = {"bf16": 0, "mxfp8": 1, "nvfp4": 2}
ACT = {"swiglu": 0, "clamped_swiglu": 1, "geglu": 2, "srelu": 3}
EXTRA_BIAS, EXTRA_SCALE = 1, 2  # moe_layer_desc_t.extras bits
DEVERR = {0: "none", 1: "capacity", 2: "timeout", 3: "bad_id"}

KERNEL_NAMES = ("route_topk", "assign_rows", "gather_x", "gemm_fc1_fprop", "gemm_fc2_fprop",
                "combine_y", "gather_dy", "gemm_fc2_dgrad", "dprob_reduce", "gemm_fc2_wgrad",
                "gemm_fc1_dgrad", "combine_dx", "gemm_fc1_wgrad", "mxfp8_quantize", "pack_fc1",
                "extras_reduce", "nvfp4_amax", "nvfp4_quantize", "route_export")
# moe_ws_layout_t.nv_amax slots (fp32 [16], first 10 used)
NV_AMAX = ("x", "xt", "w1", "w2", "a", "at", "dy", "dyt", "dz", "dzt")

EXPORTS = ("moe_timeline_begin", "moe_timeline_end", "moe_workspace_size", "moe_workspace_layout", "moe_route_permute",
           "moe_grouped_mlp_fwd", "moe_grouped_mlp_bwd", "mxfp8_quantize", "moe_pack_fc1_weight",
           "moe_get_error", "moe_clear_error", "moe_gemm_ctas", "moe_launch_count",
           "moe_last_error_string", "moe_selftest_wait_timeout", "moe_selftest_gemm_timeout",
           "moe_route_export",
           "moe_grouped_mlp_fwd_ex",
           "moe_grouped_mlp_bwd_ex", "nvfp4_amax", "nvfp4_quantize")


class LayerDesc(ctypes.Structure):
    _fields_ = [("E", ctypes.c_int32), ("k", ctypes.c_int32), ("H", ctypes.c_int32),
                ("F", ctypes.c_int32), ("T_max", ctypes.c_int32), ("precision", ctypes.c_int32),
                ("activation", ctypes.c_int32), ("beta", ctypes.c_float),
                ("gate_max", ctypes.c_float), ("lin_lo", ctypes.c_float),
                ("lin_hi", ctypes.c_float), ("lin_offset", ctypes.c_float),
                ("sm_margin", ctypes.c_int32), ("ilv", ctypes.c_int32), ("align", ctypes.c_int32),
                ("recompute", ctypes.c_int32), ("extras", ctypes.c_int32),
                ("rht_mask", ctypes.c_uint32), ("reuse_weights", ctypes.c_int32),
                ("pdl", ctypes.c_int32)]


class WsLayout(ctypes.Structure):
    _fields_ = [("total", ctypes.c_size_t), ("R_cap", ctypes.c_int64), ("err", ctypes.c_size_t),
                ("offsets", ctypes.c_size_t), ("row_of", ctypes.c_size_t),
                ("src_of", ctypes.c_size_t), ("row_prob", ctypes.c_size_t),
                ("x_perm", ctypes.c_size_t), ("z", ctypes.c_size_t), ("a_s", ctypes.c_size_t),
                ("y_perm", ctypes.c_size_t), ("dy_perm", ctypes.c_size_t),
                ("dz", ctypes.c_size_t), ("dx_perm", ctypes.c_size_t),
                ("dprob_part", ctypes.c_size_t), ("ext_part", ctypes.c_size_t),
                ("mx_base", ctypes.c_size_t), ("nv_amax", ctypes.c_size_t),
                ("nv_base", ctypes.c_size_t)]


_lib = None
_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_DP = ctypes.POINTER(LayerDesc)


def load():
    """Load the shared library (build it first with __graft_entry__.build() or
    `python -m grouped_gemm_device_gb300.build`). Raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libmoegmm.so not built ({LIB_PATH}); run the build step first")
    lib = ctypes.CDLL(LIB_PATH)
    sig = {
        "moe_workspace_size": (_SZ, [_DP]),
        "moe_workspace_layout": (_I32, [_DP, ctypes.POINTER(WsLayout)]),
        "moe_route_permute": (_I32, [_DP, _I32, _P, _P, _P, _P, _P, _P, _SZ, _P]),
        "moe_grouped_mlp_fwd": (_I32, [_DP, _I32, _P, _P, _P, _P, _SZ, _P]),
        "moe_grouped_mlp_bwd": (_I32, [_DP, _I32, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
        "mxfp8_quantize": (_I32, [_P, _I64, _I64, _I32, _I32, _P, _I32, _P, _P, _P, _P, _P]),
        "nvfp4_amax": (_I32, [_P, _I64, _I64, ctypes.c_uint32, _P, _P, _P]),
        "nvfp4_quantize": (_I32, [_P, _I64, _I64, _P, _P, _I32, ctypes.c_uint32, _P, _P, _P, _P,
                                  _P]),
        "moe_pack_fc1_weight": (_I32, [_P, _P, _I32, _I32, _I32, _I32, _I32, _I32, _P]),
        "moe_get_error": (_I32, [_DP, _P, ctypes.POINTER(_I32), _P]),
        "moe_clear_error": (_I32, [_DP, _P, _P]),
        "moe_gemm_ctas": (_I32, [_DP]),
        "moe_launch_count": (ctypes.c_uint64, []),
        "moe_last_error_string": (ctypes.c_char_p, []),
        "moe_timeline_begin": (_I32, [ctypes.POINTER(_P), _I32]),
        "moe_timeline_end": (_I32, [ctypes.POINTER(_I32)]),
        "moe_route_permute_noalloc": (_I32, [_DP, _I32, _P, _P, _P, _P, _P, _P, _P, _I64, _P]),
        "moe_selftest_wait_timeout": (_I32, [_P, ctypes.c_uint64, _P]),
        "moe_selftest_gemm_timeout": (_I32, [_DP, _P, _SZ, _P, ctypes.c_uint64, _P]),
        "moe_route_export": (_I32, [_DP, _P, _SZ, _I32, _P, _P, _P, _P, _P]),
        "moe_grouped_mlp_fwd_ex": (_I32, [_DP, _I32, _P, _P, _P, _P, _P, _P, _SZ, _P]),
        "moe_grouped_mlp_bwd_ex": (_I32, [_DP, _I32, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                          _SZ, _P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


class MoeError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"status {status}: {msg}")
        self.status = status


def _check(st: int):
    if st != 0:
        raise MoeError(st, load().moe_last_error_string().decode())


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def make_desc(E, k, H, F, T_max, precision="bf16", activation="swiglu", beta=1.0,
              gate_max=math.inf, lin_lo=-math.inf, lin_hi=math.inf, lin_offset=0.0,
              sm_margin=0, ilv=64, align=32, recompute=False, extras=0,
              rht_mask=0, reuse_weights=False, pdl=False) -> LayerDesc:
    """extras: bit 0 FC1 bias, bit 1 feature scale (EXTRA_BIAS | EXTRA_SCALE). rht_mask: the
    16 signs of the NVFP4 weight-gradient rotation (bit j set: row j of a block negated).
    reuse_weights: the forward reuses the workspace's block-scaled weight copies. pdl: launch
    the call's kernels with programmatic stream serialization."""
    return LayerDesc(E, k, H, F, T_max, PREC[precision], ACT[activation], beta, gate_max,
                     lin_lo, lin_hi, lin_offset, sm_margin, ilv, align, int(recompute),
                     int(extras), int(rht_mask) & 0xFFFF, int(reuse_weights), int(pdl))


def desc_from_config(cfg, T_max=None, sm_margin=0, recompute=False, extras=0,
                     rht_mask=None) -> LayerDesc:
    """A description of a synthetic workload (synth.LayerConfig); an NVFP4 layer takes the
    workload's seeded rotation signs unless rht_mask is given."""
    if rht_mask is None:
        from . import synth
        rht_mask = synth.gen_rht_mask(cfg) if cfg.precision == "nvfp4" else 0
    return make_desc(cfg.E, cfg.k, cfg.H, cfg.F, cfg.T if T_max is None else T_max,
                     cfg.precision, cfg.activation, cfg.beta, cfg.gate_max, cfg.lin_lo,
                     cfg.lin_hi, cfg.lin_offset, sm_margin, cfg.ilv, cfg.align, recompute,
                     extras, rht_mask)


# ------------------------------------------------------------------ C ABI, same names
def moe_workspace_size(desc: LayerDesc) -> int:
    n = load().moe_workspace_size(ctypes.byref(desc))
    if n == 0:
        raise MoeError(1, load().moe_last_error_string().decode())
    return n


def moe_workspace_layout(desc: LayerDesc) -> WsLayout:
    out = WsLayout()
    _check(load().moe_workspace_layout(ctypes.byref(desc), ctypes.byref(out)))
    return out


def moe_route_permute(desc, T, logits, x, topk_ids, topk_probs, counts, ws, ws_bytes,
                      stream=None):
    _check(load().moe_route_permute(ctypes.byref(desc), T, _ptr(logits), _ptr(x), _ptr(topk_ids),
                                    _ptr(topk_probs), _ptr(counts), _ptr(ws), ws_bytes,
                                    _stream(stream)))


def moe_route_permute_noalloc(desc, T, logits, x, topk_ids, topk_probs, counts, offsets,
                              x_perm, x_perm_rows, stream=None):
    """Route + permute into caller buffers with no workspace and no device allocation (the
    library keeps its small scratch in a static device array; see include/moegmm.h)."""
    _check(load().moe_route_permute_noalloc(ctypes.byref(desc), T, _ptr(logits), _ptr(x),
                                            _ptr(topk_ids), _ptr(topk_probs), _ptr(counts),
                                            _ptr(offsets), _ptr(x_perm), x_perm_rows,
                                            _stream(stream)))


def moe_grouped_mlp_fwd(desc, T, w1_packed, w2, y, ws, ws_bytes, stream=None):
    _check(load().moe_grouped_mlp_fwd(ctypes.byref(desc), T, _ptr(w1_packed), _ptr(w2), _ptr(y),
                                      _ptr(ws), ws_bytes, _stream(stream)))


def moe_grouped_mlp_bwd(desc, T, dy, w1_packed, w2, dx, dw1_packed, dw2, d_probs, ws, ws_bytes,
                        stream=None):
    _check(load().moe_grouped_mlp_bwd(ctypes.byref(desc), T, _ptr(dy), _ptr(w1_packed), _ptr(w2),
                                      _ptr(dx), _ptr(dw1_packed), _ptr(dw2), _ptr(d_probs),
                                      _ptr(ws), ws_bytes, _stream(stream)))


def moe_grouped_mlp_fwd_ex(desc, T, w1_packed, w2, fc1_bias, feat_scale, y, ws, ws_bytes,
                           stream=None):
    _check(load().moe_grouped_mlp_fwd_ex(ctypes.byref(desc), T, _ptr(w1_packed), _ptr(w2),
                                         _ptr(fc1_bias), _ptr(feat_scale), _ptr(y), _ptr(ws),
                                         ws_bytes, _stream(stream)))


def moe_grouped_mlp_bwd_ex(desc, T, dy, w1_packed, w2, feat_scale, dx, dw1_packed, dw2, d_probs,
                           d_fc1_bias, d_feat_scale, ws, ws_bytes, stream=None):
    _check(load().moe_grouped_mlp_bwd_ex(ctypes.byref(desc), T, _ptr(dy), _ptr(w1_packed),
                                         _ptr(w2), _ptr(feat_scale), _ptr(dx), _ptr(dw1_packed),
                                         _ptr(dw2), _ptr(d_probs), _ptr(d_fc1_bias),
                                         _ptr(d_feat_scale), _ptr(ws), ws_bytes, _stream(stream)))


def mxfp8_quantize(inp, M, N, rowwise, colwise, q_row=None, s_row=None, q_col=None, s_col=None,
                   stream=None, group_offsets=None, num_groups=0):
    """group_offsets: int32 device tensor [num_groups + 1]; column-wise blocks then restart at
    each group's first row and s_col is [N, mxfp8_grouped_scale_cols(M, num_groups)]."""
    _check(load().mxfp8_quantize(_ptr(inp), M, N, int(rowwise), int(colwise),
                                 _ptr(group_offsets), int(num_groups), _ptr(q_row), _ptr(s_row),
                                 _ptr(q_col), _ptr(s_col), _stream(stream)))


def mxfp8_grouped_scale_cols(M, num_groups) -> int:
    """Entries per column of the grouped column-wise scales (include/moegmm.h)."""
    return 4 * ((-(-M // 32) + num_groups + 3) // 4)


def nvfp4_amax(inp, M, N, sign_mask, amax, amax_rht=None, stream=None):
    _check(load().nvfp4_amax(_ptr(inp), M, N, int(sign_mask) & 0xFFFF, _ptr(amax),
                             _ptr(amax_rht), _stream(stream)))


def nvfp4_quantize(inp, M, N, amax_row, amax_col, rht, sign_mask, q_row=None, s_row=None,
                   q_col=None, s_col=None, stream=None):
    _check(load().nvfp4_quantize(_ptr(inp), M, N, _ptr(amax_row), _ptr(amax_col), int(rht),
                                 int(sign_mask) & 0xFFFF, _ptr(q_row), _ptr(s_row), _ptr(q_col),
                                 _ptr(s_col), _stream(stream)))


def moe_pack_fc1_weight(src, dst, E, H, F, gated, ilv, inverse, stream=None):
    _check(load().moe_pack_fc1_weight(_ptr(src), _ptr(dst), E, H, F, int(gated), ilv,
                                      int(inverse), _stream(stream)))


def moe_selftest_wait_timeout(err, limit_ns, stream=None):
    """Enqueue the bounded-wait self-test: a wait nothing completes gives up after limit_ns
    and writes the timeout code into the device int32 `err`."""
    _check(load().moe_selftest_wait_timeout(_ptr(err), int(limit_ns), _stream(stream)))


def moe_selftest_gemm_timeout(desc, ws, ws_bytes, w2, limit_ns, stream=None):
    """Enqueue the FC2 forward GEMM of a routed BF16 layer with its loads withheld: every wait
    of the kernel runs out after limit_ns and the workspace error word records the timeout."""
    _check(load().moe_selftest_gemm_timeout(ctypes.byref(desc), _ptr(ws), ws_bytes, _ptr(w2),
                                            int(limit_ns), _stream(stream)))


def moe_route_export(desc, ws, ws_bytes, T, offsets=None, row_of=None, src_of=None,
                     row_prob=None, stream=None):
    """Copy the routing maps of the last route on ws into caller tensors (any may be None)."""
    _check(load().moe_route_export(ctypes.byref(desc), _ptr(ws), ws_bytes, int(T),
                                   _ptr(offsets), _ptr(row_of), _ptr(src_of), _ptr(row_prob),
                                   _stream(stream)))


def moe_get_error(desc, ws, stream=None) -> int:
    """Synchronous convenience: enqueue the copy, synchronise the stream, return the code."""
    import torch
    code = ctypes.c_int32(-1)
    _check(load().moe_get_error(ctypes.byref(desc), _ptr(ws), ctypes.byref(code),
                                _stream(stream)))
    torch.cuda.synchronize()
    return code.value


def moe_clear_error(desc, ws, stream=None):
    _check(load().moe_clear_error(ctypes.byref(desc), _ptr(ws), _stream(stream)))


def moe_gemm_ctas(desc) -> int:
    return load().moe_gemm_ctas(ctypes.byref(desc))


def moe_launch_count() -> int:
    return int(load().moe_launch_count())


class Timeline:
    """Records a CUDA event after every library kernel launch (moe_timeline_begin/end) and
    turns consecutive event pairs into per-kernel durations."""

    def __init__(self, capacity: int):
        import torch
        self.capacity = capacity
        self.events = [torch.cuda.Event(enable_timing=True) for _ in range(capacity)]
        for e in self.events:           # torch creates events lazily: force creation
            e.record()
        torch.cuda.synchronize()
        self._handles = (_P * capacity)(*[e.cuda_event for e in self.events])
        self.ids = []

    def begin(self):
        _check(load().moe_timeline_begin(self._handles, self.capacity))

    def end(self) -> int:
        buf = (_I32 * self.capacity)()
        n = load().moe_timeline_end(buf)
        self.ids = list(buf[:n])
        return n

    def durations(self, start_event):
        """[(kernel_name, ms)] for each recorded launch, after a synchronize."""
        out = []
        prev = start_event
        for i, kid in enumerate(self.ids):
            out.append((KERNEL_NAMES[kid], prev.elapsed_time(self.events[i])))
            prev = self.events[i]
        return out


# ------------------------------------------------------------------ buffer plumbing
class MoELayer:
    """Owns the caller-side buffers of one layer (allocated with torch) and runs the C ABI
    calls on them. Weights: w1_packed [E, N1, H] bf16 (packed rows), w2 [E, F, H] bf16."""

    def __init__(self, desc: LayerDesc, device="cuda"):
        import torch
        load()
        self.desc = desc
        self.device = torch.device(device)
        self.layout = moe_workspace_layout(desc)
        self.ws_bytes = self.layout.total
        self.ws = torch.zeros(self.ws_bytes, dtype=torch.uint8, device=self.device)
        d = desc
        self.N1 = d.F if d.activation == ACT["srelu"] else 2 * d.F
        T, E, k, H = d.T_max, d.E, d.k, d.H
        dev = self.device
        self.topk_ids = torch.empty(T, k, dtype=torch.int32, device=dev)
        self.topk_probs = torch.empty(T, k, dtype=torch.float32, device=dev)
        self.counts = torch.zeros(E, dtype=torch.int32, device=dev)
        self.y = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
        self.dx = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
        self.d_probs = torch.empty(T, k, dtype=torch.float32, device=dev)
        self.dw1 = None
        self.dw2 = None
        self.d_fc1_bias = None     # extras: [E, N1] fp32, logical order
        self.d_feat_scale = None   # extras: [E, F] fp32

    # views into the workspace -------------------------------------------------------
    def ws_view(self, name, dtype, shape):
        import torch
        off = getattr(self.layout, name)
        n = 1
        for s in shape:
            n *= s
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        return self.ws[off:off + nbytes].view(dtype).view(*shape)

    def offsets(self):
        import torch
        return self.ws_view("offsets", torch.int32, (self.desc.E + 1,))

    # calls ---------------------------------------------------------------------------
    def route_permute(self, logits, x, T=None, stream=None):
        T = logits.shape[0] if T is None else T
        moe_route_permute(self.desc, T, logits, x, self.topk_ids, self.topk_probs, self.counts,
                          self.ws, self.ws_bytes, stream)

    def forward(self, w1_packed, w2, T, stream=None, fc1_bias=None, feat_scale=None):
        """fc1_bias fp32 [E, N1] (logical order) and feat_scale fp32 [E, F] for a layer made
        with the matching extras bits."""
        if self.desc.extras:
            moe_grouped_mlp_fwd_ex(self.desc, T, w1_packed, w2, fc1_bias, feat_scale, self.y,
                                   self.ws, self.ws_bytes, stream)
        else:
            moe_grouped_mlp_fwd(self.desc, T, w1_packed, w2, self.y, self.ws, self.ws_bytes,
                                stream)
        return self.y[:T]

    def backward(self, dy, w1_packed, w2, T, stream=None, feat_scale=None):
        import torch
        if self.dw1 is None:
            d = self.desc
            self.dw1 = torch.empty(d.E, self.N1, d.H, dtype=torch.bfloat16, device=self.device)
            self.dw2 = torch.empty(d.E, d.F, d.H, dtype=torch.bfloat16, device=self.device)
        if self.desc.extras:
            if self.d_fc1_bias is None:
                d = self.desc
                self.d_fc1_bias = (torch.empty(d.E, self.N1, dtype=torch.float32,
                                               device=self.device) if d.extras & 1 else None)
                self.d_feat_scale = (torch.empty(d.E, d.F, dtype=torch.float32,
                                                 device=self.device) if d.extras & 2 else None)
            moe_grouped_mlp_bwd_ex(self.desc, T, dy, w1_packed, w2, feat_scale, self.dx,
                                   self.dw1, self.dw2, self.d_probs, self.d_fc1_bias,
                                   self.d_feat_scale, self.ws, self.ws_bytes, stream)
        else:
            moe_grouped_mlp_bwd(self.desc, T, dy, w1_packed, w2, self.dx, self.dw1, self.dw2,
                                self.d_probs, self.ws, self.ws_bytes, stream)
        return self.dx[:T], self.dw1, self.dw2, self.d_probs[:T]

    def device_error(self, stream=None) -> int:
        return moe_get_error(self.desc, self.ws, stream)


def pack_w1(w1_logical, gated=True, ilv=64, stream=None):
    """w1_logical bf16 [E, H, N1] (torch, cuda) -> packed [E, N1, H] through the library."""
    import torch
    E, H, N1 = w1_logical.shape
    F = N1 // 2 if gated else N1
    out = torch.empty(E, N1, H, dtype=w1_logical.dtype, device=w1_logical.device)
    moe_pack_fc1_weight(w1_logical, out, E, H, F, gated, ilv, 0, stream)
    return out
