"""Python binding of the flint_moe C ABI (include/flint_moe.h).

Argument marshalling only: every step of the layer runs in the CUDA kernels of
``libflint_moe.so``.  PyTorch supplies device memory and streams.  There is no fallback:
if the library is missing or the device is not an sm_103 GPU, the calls raise.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_NAME = "libflint_moe.so"

HIDDEN, N_EXPERTS, TOP_K, EXPERT_INTER, SHARED_INTER = 2048, 256, 6, 512, 1024
FLAG_PRE_RMSNORM = 0x1
FLAG_RESIDUAL = 0x2
FLAG_TEST_WAIT_TIMEOUT = 0x80000000  # tests of the device-timeout path only
TRACE_SLOTS = 24  # trace values per CTA (flint_moe_read_trace)

STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "workspace", 4: "cuda error",
          5: "device timeout", 6: "device bounds"}

# Every entry point declared in include/flint_moe.h.
EXPORTS = ("flint_moe_status_string", "flint_moe_workspace_bytes", "flint_moe_create", "flint_moe_route",
           "flint_moe_forward", "flint_moe_forward_host", "flint_moe_poll_device_status",
           "flint_moe_enable_kernel_timing", "flint_moe_kernel_times", "flint_moe_read_trace",
           "flint_moe_destroy", "flint_moe_forward_noalloc", "flint_moe_noalloc_poll_device_status",
           "flint_moe_stack_workspace_bytes",
           "flint_moe_stack_create", "flint_moe_stack_forward", "flint_moe_stack_poll_device_status",
           "flint_moe_stack_enable_kernel_timing", "flint_moe_stack_read_trace", "flint_moe_stack_destroy",
           "flint_dense_workspace_bytes", "flint_dense_create", "flint_dense_forward",
           "flint_dense_poll_device_status", "flint_dense_enable_kernel_timing", "flint_dense_kernel_times",
           "flint_dense_destroy", "flint_swa_workspace_bytes", "flint_swa_workspace_init", "flint_swa_decode",
           "flint_swa_poll_device_status", "flint_moe_create_nvfp4")

NOALLOC_MAX_TOKENS = 4
DENSE_INTER = 6144  # width of the dense MLP layers


class FlintMoEError(RuntimeError):
    def __init__(self, code, what):
        self.code = code
        super().__init__(f"{what}: {STATUS.get(code, code)}")


class _Config(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int), ("n_experts", ctypes.c_int), ("top_k", ctypes.c_int),
                ("expert_inter", ctypes.c_int), ("shared_inter", ctypes.c_int), ("max_tokens", ctypes.c_int),
                ("flags", ctypes.c_uint), ("rms_eps", ctypes.c_float)]


class _DenseConfig(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int), ("inter", ctypes.c_int), ("max_tokens", ctypes.c_int),
                ("flags", ctypes.c_uint), ("rms_eps", ctypes.c_float)]


class _DenseWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("w_gate", "w_up", "w_down")]


class _Nvfp4Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("w_router", "router_bias", "gate_codes", "up_codes", "down_codes", "gate_scales", "up_scales",
                 "down_scales", "gate_tscale", "up_tscale", "down_tscale", "sgate_codes", "sup_codes",
                 "sdown_codes", "sgate_scales", "sup_scales", "sdown_scales")] + \
               [("sgate_tscale", ctypes.c_float), ("sup_tscale", ctypes.c_float), ("sdown_tscale", ctypes.c_float)]


class _Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("w_router", "router_bias", "w_gate", "w_up", "w_down", "ws_gate", "ws_up", "ws_down")]


_LIB = None


def lib_path() -> str:
    return os.path.join(_HERE, LIB_NAME)


def load_library():
    """Load libflint_moe.so (raises if it has not been built)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = lib_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with __graft_entry__.build() "
                           "(python -m sparse_moe_layer_15_b300.build)")
    L = ctypes.CDLL(path)
    P, I32 = ctypes.c_void_p, ctypes.c_int
    L.flint_moe_status_string.argtypes = [I32]
    L.flint_moe_status_string.restype = ctypes.c_char_p
    L.flint_moe_workspace_bytes.argtypes = [ctypes.POINTER(_Config), ctypes.POINTER(ctypes.c_size_t)]
    L.flint_moe_create.argtypes = [ctypes.POINTER(_Config), ctypes.POINTER(_Weights), P, ctypes.c_size_t,
                                   ctypes.POINTER(P)]
    L.flint_moe_route.argtypes = [P, P, I32, P, P, P, P]
    L.flint_moe_forward.argtypes = [P, P, I32, P, P, P, P]
    L.flint_moe_forward_host.argtypes = [P, P, I32, P, P]
    L.flint_moe_poll_device_status.argtypes = [P, P]
    L.flint_moe_enable_kernel_timing.argtypes = [P, I32]
    L.flint_moe_kernel_times.argtypes = [P, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(ctypes.c_float), I32,
                                         ctypes.POINTER(I32)]
    L.flint_moe_read_trace.argtypes = [P, ctypes.POINTER(ctypes.c_ulonglong), I32, ctypes.POINTER(I32)]
    L.flint_moe_destroy.argtypes = [P]
    L.flint_moe_forward_noalloc.argtypes = [ctypes.POINTER(_Weights), P, I32, P, P, P, P]
    L.flint_moe_noalloc_poll_device_status.argtypes = [P]
    L.flint_moe_stack_workspace_bytes.argtypes = [ctypes.POINTER(_Config), I32, ctypes.POINTER(ctypes.c_size_t)]
    L.flint_moe_stack_create.argtypes = [ctypes.POINTER(_Config), ctypes.POINTER(_Weights), I32, P, ctypes.c_size_t,
                                         ctypes.POINTER(P)]
    L.flint_moe_stack_forward.argtypes = [P, P, I32, P, P, P]
    L.flint_moe_stack_poll_device_status.argtypes = [P, P]
    L.flint_moe_stack_enable_kernel_timing.argtypes = [P, I32]
    L.flint_moe_stack_read_trace.argtypes = [P, ctypes.POINTER(ctypes.c_ulonglong), I32, ctypes.POINTER(I32)]
    L.flint_moe_stack_destroy.argtypes = [P]
    L.flint_dense_workspace_bytes.argtypes = [ctypes.POINTER(_DenseConfig), ctypes.POINTER(ctypes.c_size_t)]
    L.flint_dense_create.argtypes = [ctypes.POINTER(_DenseConfig), ctypes.POINTER(_DenseWeights), P,
                                     ctypes.c_size_t, ctypes.POINTER(P)]
    L.flint_dense_forward.argtypes = [P, P, I32, P, P]
    L.flint_dense_poll_device_status.argtypes = [P, P]
    L.flint_dense_enable_kernel_timing.argtypes = [P, I32]
    L.flint_dense_kernel_times.argtypes = [P, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(ctypes.c_float), I32,
                                           ctypes.POINTER(I32)]
    L.flint_dense_destroy.argtypes = [P]
    L.flint_moe_create_nvfp4.argtypes = [ctypes.POINTER(_Config), ctypes.POINTER(_Nvfp4Weights), P, ctypes.c_size_t,
                                         ctypes.POINTER(P)]
    L.flint_swa_workspace_bytes.argtypes = [I32, ctypes.POINTER(ctypes.c_size_t)]
    L.flint_swa_workspace_init.argtypes = [P, ctypes.c_size_t, P]
    L.flint_swa_decode.argtypes = [P, ctypes.c_size_t, P, P, P, P, P, I32, P, P]
    L.flint_swa_poll_device_status.argtypes = [P, P]
    for name in EXPORTS:
        if name != "flint_moe_status_string":
            getattr(L, name).restype = I32
    _LIB = L
    return L


def _check(rc, what):
    if rc != 0:
        raise FlintMoEError(rc, what)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_ptr(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def workspace_bytes(max_tokens: int, flags: int = 0, rms_eps: float = 1e-6) -> int:
    L = load_library()
    cfg = _Config(HIDDEN, N_EXPERTS, TOP_K, EXPERT_INTER, SHARED_INTER, max_tokens, flags, rms_eps)
    n = ctypes.c_size_t(0)
    _check(L.flint_moe_workspace_bytes(ctypes.byref(cfg), ctypes.byref(n)), "flint_moe_workspace_bytes")
    return n.value


def forward_noalloc(weights: dict, x, y=None, topk_idx=None, topk_w=None, stream=None):
    """The whole layer through flint_moe_forward_noalloc: no workspace, no allocation by the
    library (for callers that cannot allocate device memory where they run the layer).
    1 <= T <= NOALLOC_MAX_TOKENS; ``weights`` as for :class:`FlintMoE`.  ``y`` is allocated
    here by torch when not given, which is the caller's choice, not the library's."""
    import torch
    L = load_library()
    T = x.shape[0]
    if y is None:
        y = torch.empty_like(x)
    w = _Weights(*[(weights[n].data_ptr() if weights.get(n) is not None else None) for n, _ in _Weights._fields_])
    _check(L.flint_moe_forward_noalloc(ctypes.byref(w), _ptr(x), T, _ptr(y), _ptr(topk_idx), _ptr(topk_w),
                                       _stream_ptr(stream)), "flint_moe_forward_noalloc")
    return y


def noalloc_poll_device_status(stream=None) -> int:
    """Status code of the allocation-free entry point's device errors on the current device
    since the last poll (0 = ok, 5 = device timeout, 6 = device bounds); clears it."""
    return load_library().flint_moe_noalloc_poll_device_status(_stream_ptr(stream))


class FlintMoE:
    """One Flint MoE layer bound to borrowed bf16 device weights.

    ``weights``: dict with torch CUDA tensors ``w_router`` [2048,256], ``w_gate``/``w_up``
    [256,2048,512], ``w_down`` [256,512,2048], ``ws_gate``/``ws_up`` [2048,1024],
    ``ws_down`` [1024,2048] (bf16, contiguous) and optionally ``router_bias`` [256] fp32.
    The tensors must stay alive as long as the layer."""

    def __init__(self, weights: dict, max_tokens: int, flags: int = 0, rms_eps: float = 1e-6,
                 workspace=None):
        import torch
        self._L = load_library()
        self.max_tokens = int(max_tokens)
        self.flags = int(flags)
        self._weights = weights  # keep the borrowed tensors alive
        for k, v in weights.items():
            if v is not None and not v.is_contiguous():
                raise ValueError(f"{k} must be contiguous")
        self._cfg = _Config(HIDDEN, N_EXPERTS, TOP_K, EXPERT_INTER, SHARED_INTER, self.max_tokens, self.flags,
                            float(rms_eps))
        self._w = _Weights(*[(weights[n].data_ptr() if weights.get(n) is not None else None)
                             for n, _ in _Weights._fields_])
        nbytes = ctypes.c_size_t(0)
        _check(self._L.flint_moe_workspace_bytes(ctypes.byref(self._cfg), ctypes.byref(nbytes)),
               "flint_moe_workspace_bytes")
        dev = weights["w_router"].device
        if workspace is None:
            workspace = torch.empty(nbytes.value, dtype=torch.uint8, device=dev)
        self.workspace = workspace
        h = ctypes.c_void_p()
        _check(self._L.flint_moe_create(ctypes.byref(self._cfg), ctypes.byref(self._w),
                                        ctypes.c_void_p(workspace.data_ptr()), workspace.numel(),
                                        ctypes.byref(h)), "flint_moe_create")
        self._h = h

    @classmethod
    def nvfp4(cls, w_router, q, max_tokens: int, router_bias=None, flags: int = 0, rms_eps: float = 1e-6,
              workspace=None):
        """A layer on NVFP4 expert weights (flint_moe_create_nvfp4; decode sizes, max_tokens <= 64).
        ``q``: name -> (codes, scales, tensor_scale) for w_gate, w_up, w_down (routed: tensor scales
        [256] fp32 on the device) and ws_gate, ws_up, ws_down (shared: scalar tensor scales), in the
        layouts of include/flint_moe.h; ``w_router`` bf16 [2048, 256].  Borrowed: keep them alive."""
        import torch
        self = cls.__new__(cls)
        self._L = load_library()
        self.max_tokens = int(max_tokens)
        self.flags = int(flags)
        self._weights = (w_router, router_bias, q)
        self._cfg = _Config(HIDDEN, N_EXPERTS, TOP_K, EXPERT_INTER, SHARED_INTER, self.max_tokens, self.flags,
                            float(rms_eps))

        def ptr(t):
            if not t.is_contiguous():
                raise ValueError("NVFP4 tensors must be contiguous")
            return t.data_ptr()

        self._w = _Nvfp4Weights(
            ptr(w_router), None if router_bias is None else ptr(router_bias),
            ptr(q["w_gate"][0]), ptr(q["w_up"][0]), ptr(q["w_down"][0]),
            ptr(q["w_gate"][1]), ptr(q["w_up"][1]), ptr(q["w_down"][1]),
            ptr(q["w_gate"][2]), ptr(q["w_up"][2]), ptr(q["w_down"][2]),
            ptr(q["ws_gate"][0]), ptr(q["ws_up"][0]), ptr(q["ws_down"][0]),
            ptr(q["ws_gate"][1]), ptr(q["ws_up"][1]), ptr(q["ws_down"][1]),
            float(q["ws_gate"][2]), float(q["ws_up"][2]), float(q["ws_down"][2]))
        nbytes = ctypes.c_size_t(0)
        _check(self._L.flint_moe_workspace_bytes(ctypes.byref(self._cfg), ctypes.byref(nbytes)),
               "flint_moe_workspace_bytes")
        if workspace is None:
            workspace = torch.empty(nbytes.value, dtype=torch.uint8, device=w_router.device)
        self.workspace = workspace
        h = ctypes.c_void_p()
        _check(self._L.flint_moe_create_nvfp4(ctypes.byref(self._cfg), ctypes.byref(self._w),
                                              ctypes.c_void_p(workspace.data_ptr()), workspace.numel(),
                                              ctypes.byref(h)), "flint_moe_create_nvfp4")
        self._h = h
        return self

    def route(self, x, topk_idx=None, topk_w=None, counts=None, stream=None):
        import torch
        T = x.shape[0]
        if topk_idx is None:
            topk_idx = torch.empty((T, TOP_K), dtype=torch.int32, device=x.device)
        if topk_w is None:
            topk_w = torch.empty((T, TOP_K), dtype=torch.float32, device=x.device)
        if counts is None:
            counts = torch.empty((N_EXPERTS,), dtype=torch.int32, device=x.device)
        _check(self._L.flint_moe_route(self._h, _ptr(x), T, _ptr(topk_idx), _ptr(topk_w), _ptr(counts),
                                       _stream_ptr(stream)), "flint_moe_route")
        return topk_idx, topk_w, counts

    def forward(self, x, y=None, topk_idx=None, topk_w=None, stream=None):
        import torch
        T = x.shape[0]
        if y is None:
            y = torch.empty_like(x)
        _check(self._L.flint_moe_forward(self._h, _ptr(x), T, _ptr(y), _ptr(topk_idx), _ptr(topk_w),
                                         _stream_ptr(stream)), "flint_moe_forward")
        return y

    def forward_host(self, x_host, y_host, stream=None):
        """x_host, y_host: CPU (ideally pinned) bf16 tensors [T, 2048]."""
        T = x_host.shape[0]
        _check(self._L.flint_moe_forward_host(self._h, ctypes.c_void_p(x_host.data_ptr()), T,
                                              ctypes.c_void_p(y_host.data_ptr()), _stream_ptr(stream)),
               "flint_moe_forward_host")
        return y_host

    def poll_device_status(self, stream=None):
        return self._L.flint_moe_poll_device_status(self._h, _stream_ptr(stream))

    def enable_kernel_timing(self, on=True):
        _check(self._L.flint_moe_enable_kernel_timing(self._h, 1 if on else 0), "flint_moe_enable_kernel_timing")

    def enable_phase_trace(self, on=True):
        _check(self._L.flint_moe_enable_kernel_timing(self._h, 2 if on else 0), "flint_moe_enable_kernel_timing")

    def read_trace(self, slots=TRACE_SLOTS):
        """The last call's trace (see flint_moe_enable_kernel_timing): list of per-CTA lists."""
        cap = 1024 * slots
        buf = (ctypes.c_ulonglong * cap)()
        n = ctypes.c_int(0)
        _check(self._L.flint_moe_read_trace(self._h, buf, cap, ctypes.byref(n)), "flint_moe_read_trace")
        return [list(buf[i:i + slots]) for i in range(0, n.value, slots)]

    def kernel_times(self):
        cap = 16
        names = (ctypes.c_char_p * cap)()
        ms = (ctypes.c_float * cap)()
        n = ctypes.c_int(0)
        _check(self._L.flint_moe_kernel_times(self._h, names, ms, cap, ctypes.byref(n)), "flint_moe_kernel_times")
        return [(names[i].decode(), float(ms[i])) for i in range(n.value)]

    def close(self):
        if getattr(self, "_h", None):
            self._L.flint_moe_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def stack_workspace_bytes(n_layers: int, max_tokens: int, flags: int = 0, rms_eps: float = 1e-6) -> int:
    L = load_library()
    cfg = _Config(HIDDEN, N_EXPERTS, TOP_K, EXPERT_INTER, SHARED_INTER, max_tokens, flags, rms_eps)
    n = ctypes.c_size_t(0)
    _check(L.flint_moe_stack_workspace_bytes(ctypes.byref(cfg), int(n_layers), ctypes.byref(n)),
           "flint_moe_stack_workspace_bytes")
    return n.value


class FlintMoEStack:
    """n MoE layers applied in place in one kernel launch (flint_moe_stack_*): x <- [x +]
    MoE_l([RMSNorm](x)) for l = 0..n-1 with the config's flags.  ``weights_list``: one dict per
    layer as for :class:`FlintMoE` (borrowed; keep them alive).  Decode sizes: max_tokens <= 256."""

    def __init__(self, weights_list, max_tokens: int, flags: int = 0, rms_eps: float = 1e-6, workspace=None):
        import torch
        self._L = load_library()
        self.n_layers = len(weights_list)
        self.max_tokens = int(max_tokens)
        self._weights = weights_list
        for w in weights_list:
            for k, v in w.items():
                if v is not None and not v.is_contiguous():
                    raise ValueError(f"{k} must be contiguous")
        self._cfg = _Config(HIDDEN, N_EXPERTS, TOP_K, EXPERT_INTER, SHARED_INTER, self.max_tokens, int(flags),
                            float(rms_eps))
        arr = (_Weights * self.n_layers)(*[
            _Weights(*[(w[n].data_ptr() if w.get(n) is not None else None) for n, _ in _Weights._fields_])
            for w in weights_list])
        nbytes = stack_workspace_bytes(self.n_layers, self.max_tokens, flags, rms_eps)
        if workspace is None:
            workspace = torch.empty(nbytes, dtype=torch.uint8, device=weights_list[0]["w_router"].device)
        self.workspace = workspace
        h = ctypes.c_void_p()
        _check(self._L.flint_moe_stack_create(ctypes.byref(self._cfg), arr, self.n_layers,
                                              ctypes.c_void_p(workspace.data_ptr()), workspace.numel(),
                                              ctypes.byref(h)), "flint_moe_stack_create")
        self._h = h

    def forward(self, x, topk_idx=None, topk_w=None, stream=None):
        """In place on x (bf16 [T, 2048] on the GPU); returns x.  topk_idx / topk_w: optional
        [n_layers, T, 6] int32 / float32 device tensors receiving every layer's routing."""
        _check(self._L.flint_moe_stack_forward(self._h, _ptr(x), x.shape[0], _ptr(topk_idx), _ptr(topk_w),
                                               _stream_ptr(stream)), "flint_moe_stack_forward")
        return x

    def poll_device_status(self, stream=None):
        return self._L.flint_moe_stack_poll_device_status(self._h, _stream_ptr(stream))

    def enable_phase_trace(self, on=True):
        _check(self._L.flint_moe_stack_enable_kernel_timing(self._h, 2 if on else 0),
               "flint_moe_stack_enable_kernel_timing")

    def read_trace(self, slots=TRACE_SLOTS):
        """The last call's phase trace (the last layer's stamps): list of per-CTA lists."""
        cap = 1024 * slots
        buf = (ctypes.c_ulonglong * cap)()
        n = ctypes.c_int(0)
        _check(self._L.flint_moe_stack_read_trace(self._h, buf, cap, ctypes.byref(n)), "flint_moe_stack_read_trace")
        return [list(buf[i:i + slots]) for i in range(0, n.value, slots)]

    def close(self):
        if getattr(self, "_h", None):
            self._L.flint_moe_stack_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class FlintDense:
    """One dense SwiGLU MLP layer (width 6144) bound to borrowed bf16 device weights:
    ``w_gate``/``w_up`` [2048, 6144], ``w_down`` [6144, 2048] (contiguous).
    y = (silu(x' Wg) * (x' Wu)) Wd [+ x] with x' = x or rms(x) (flags as for FlintMoE)."""

    def __init__(self, weights: dict, max_tokens: int, flags: int = 0, rms_eps: float = 1e-6, workspace=None):
        import torch
        self._L = load_library()
        self.max_tokens = int(max_tokens)
        self._weights = weights
        for k, v in weights.items():
            if not v.is_contiguous():
                raise ValueError(f"{k} must be contiguous")
        self._cfg = _DenseConfig(HIDDEN, DENSE_INTER, self.max_tokens, int(flags), float(rms_eps))
        self._w = _DenseWeights(*[weights[n].data_ptr() for n, _ in _DenseWeights._fields_])
        nbytes = ctypes.c_size_t(0)
        _check(self._L.flint_dense_workspace_bytes(ctypes.byref(self._cfg), ctypes.byref(nbytes)),
               "flint_dense_workspace_bytes")
        if workspace is None:
            workspace = torch.empty(nbytes.value, dtype=torch.uint8, device=weights["w_gate"].device)
        self.workspace = workspace
        h = ctypes.c_void_p()
        _check(self._L.flint_dense_create(ctypes.byref(self._cfg), ctypes.byref(self._w),
                                          ctypes.c_void_p(workspace.data_ptr()), workspace.numel(),
                                          ctypes.byref(h)), "flint_dense_create")
        self._h = h

    def forward(self, x, y=None, stream=None):
        import torch
        if y is None:
            y = torch.empty_like(x)
        _check(self._L.flint_dense_forward(self._h, _ptr(x), x.shape[0], _ptr(y), _stream_ptr(stream)),
               "flint_dense_forward")
        return y

    def poll_device_status(self, stream=None):
        return self._L.flint_dense_poll_device_status(self._h, _stream_ptr(stream))

    def enable_kernel_timing(self, on=True):
        _check(self._L.flint_dense_enable_kernel_timing(self._h, 1 if on else 0), "flint_dense_enable_kernel_timing")

    def kernel_times(self):
        cap = 16
        names = (ctypes.c_char_p * cap)()
        ms = (ctypes.c_float * cap)()
        n = ctypes.c_int(0)
        _check(self._L.flint_dense_kernel_times(self._h, names, ms, cap, ctypes.byref(n)), "flint_dense_kernel_times")
        return [(names[i].decode(), float(ms[i])) for i in range(n.value)]

    def close(self):
        if getattr(self, "_h", None):
            self._L.flint_dense_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


SWA_HEADS, SWA_KV_HEADS, SWA_HEAD_DIM, SWA_WINDOW = 32, 4, 128, 513


class SwaAttention:
    """Decode attention of the sliding-window layers (flint_swa_*): 32 query heads, 4 KV heads,
    head dimension 128, a ring of 513 cached tokens per sequence, one learned sink per head.
    The workspace is allocated here by torch (for up to ``max_batch`` sequences) and
    initialised once."""

    def __init__(self, max_batch: int, device="cuda", stream=None):
        import torch
        self._L = load_library()
        n = ctypes.c_size_t(0)
        _check(self._L.flint_swa_workspace_bytes(int(max_batch), ctypes.byref(n)), "flint_swa_workspace_bytes")
        self.workspace = torch.empty(n.value, dtype=torch.uint8, device=device)
        _check(self._L.flint_swa_workspace_init(_ptr(self.workspace), n.value, _stream_ptr(stream)),
               "flint_swa_workspace_init")

    def decode(self, q, k_cache, v_cache, sinks, pos, out=None, stream=None):
        """q [B,32,128] bf16, k_cache / v_cache [B,513,4,128] bf16, sinks [32] fp32, pos [B] int32
        (device tensors) -> out [B,32,128] bf16."""
        import torch
        if out is None:
            out = torch.empty_like(q)
        for t in (q, k_cache, v_cache, sinks, pos, out):
            if not t.is_contiguous():
                raise ValueError("flint_swa_decode takes contiguous tensors")
        _check(self._L.flint_swa_decode(_ptr(self.workspace), self.workspace.numel(), _ptr(q), _ptr(k_cache),
                                        _ptr(v_cache), _ptr(sinks), _ptr(pos), q.shape[0], _ptr(out),
                                        _stream_ptr(stream)), "flint_swa_decode")
        return out

    def poll_device_status(self, stream=None):
        return self._L.flint_swa_poll_device_status(_ptr(self.workspace), _stream_ptr(stream))
