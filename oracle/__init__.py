"""ctypes wrapper of the fp64 CPU oracle (oracle.c).

TEST INFRASTRUCTURE ONLY: the test suite, the package smoke check and the benchmark's
CPU-baseline / reference leg are the only users.  The product library never imports
this module.  See oracle.h for the definition it computes and the readings it takes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = None

_P = ctypes.c_void_p
_u16pp = ctypes.POINTER(ctypes.c_void_p)


class _Layer(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int), ("E", ctypes.c_int), ("k", ctypes.c_int),
                ("I", ctypes.c_int), ("Is", ctypes.c_int),
                ("w_router", _P), ("router_bias", _P),
                ("w_gate", _u16pp), ("w_up", _u16pp), ("w_down", _u16pp),
                ("ws_gate", _P), ("ws_up", _P), ("ws_down", _P)]


def lib_path() -> str:
    return os.path.join(_HERE, "liboracle.so")


def build(verbose: bool = False) -> str:
    src = os.path.join(_HERE, "oracle.c")
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-o", lib_path(), src, "-lm"]
    if verbose:
        print(" ".join(cmd))
    subprocess.check_call(cmd)
    return lib_path()


def _lib():
    global _LIB
    if _LIB is None:
        src = os.path.join(_HERE, "oracle.c")
        if (not os.path.exists(lib_path())) or os.path.getmtime(lib_path()) < os.path.getmtime(src):
            build()
        L = ctypes.CDLL(lib_path())
        L.oracle_router.argtypes = [_P, ctypes.c_int, ctypes.c_int, ctypes.c_int, _P, _P, _P, _P]
        L.oracle_select.argtypes = [_P, ctypes.c_int, ctypes.c_int, _P, _P, _P]
        L.oracle_swiglu.argtypes = [_P, ctypes.c_int, ctypes.c_int, _P, _P, _P, _P, _P]
        L.oracle_swiglu.restype = None
        L.oracle_moe_forward.argtypes = [ctypes.POINTER(_Layer), _P, ctypes.c_int, _P, _P, _P, _P, _P]
        L.oracle_moe_forward_given.argtypes = [ctypes.POINTER(_Layer), _P, ctypes.c_int, _P, _P]
        L.oracle_permute.argtypes = [_P, ctypes.c_int, ctypes.c_int, ctypes.c_int, _P, _P, _P, _P]
        L.oracle_rmsnorm.argtypes = [_P, ctypes.c_int, ctypes.c_int, ctypes.c_double, _P]
        L.oracle_rmsnorm.restype = None
        L.oracle_round_bf16.argtypes = [ctypes.c_double]
        L.oracle_round_bf16.restype = ctypes.c_double
        L.oracle_swa_decode.argtypes = [_P, _P, _P, _P, _P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_int, _P]
        L.oracle_e2m1_to_f64.argtypes = [ctypes.c_uint]
        L.oracle_e2m1_to_f64.restype = ctypes.c_double
        L.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint]
        L.oracle_e4m3_to_f64.restype = ctypes.c_double
        L.oracle_nvfp4_dequant.argtypes = [_P, _P, ctypes.c_float, ctypes.c_int, ctypes.c_int, _P]
        L.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        L.oracle_bf16_to_f64.restype = ctypes.c_double
        _LIB = L
    return _LIB


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check(rc, what):
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


def _u16(a):
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("bf16 arrays are passed as uint16 bit patterns")
    return a


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def bf16_to_f64(bits) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float64."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


class Layer:
    """One MoE layer's weights as bf16 bit arrays (uint16), for the oracle.

    ``w_gate``/``w_up``/``w_down`` are either full arrays ([E,H,I], [E,H,I], [E,I,H]) or
    dicts {expert: array} holding only some experts (a token routed to a missing expert
    makes the oracle raise)."""

    def __init__(self, w_router, w_gate, w_up, w_down, ws_gate, ws_up, ws_down,
                 router_bias=None, k=6):
        self.w_router = _u16(w_router)
        H, E = self.w_router.shape
        self.H, self.E, self.k = H, E, k
        self.router_bias = None if router_bias is None else np.ascontiguousarray(router_bias, dtype=np.float32)
        self.ws_gate, self.ws_up, self.ws_down = _u16(ws_gate), _u16(ws_up), _u16(ws_down)
        self.Is = self.ws_gate.shape[1]

        def experts(w):
            if isinstance(w, dict):
                return {int(e): _u16(v) for e, v in w.items()}
            w = _u16(w)
            return {e: w[e] for e in range(E)}

        self.w_gate, self.w_up, self.w_down = experts(w_gate), experts(w_up), experts(w_down)
        any_e = next(iter(self.w_gate.values()))
        self.I = any_e.shape[1]
        arr = ctypes.c_void_p * E

        def ptrs(d):
            return arr(*[(d[e].ctypes.data if e in d else None) for e in range(E)])

        self._pg, self._pu, self._pd = ptrs(self.w_gate), ptrs(self.w_up), ptrs(self.w_down)
        self._c = _Layer(H, E, k, self.I, self.Is, self.w_router.ctypes.data,
                         None if self.router_bias is None else self.router_bias.ctypes.data,
                         ctypes.cast(self._pg, _u16pp), ctypes.cast(self._pu, _u16pp),
                         ctypes.cast(self._pd, _u16pp), self.ws_gate.ctypes.data,
                         self.ws_up.ctypes.data, self.ws_down.ctypes.data)


def router(x, w_router, bias=None):
    """(logits, scores) in float64 for rows x ([T,H] float64)."""
    x = _f64(x)
    w_router = _u16(w_router)
    T, H = x.shape
    E = w_router.shape[1]
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    lg = np.empty((T, E))
    s = np.empty((T, E))
    _check(_lib().oracle_router(_ptr(x), T, H, E, _ptr(w_router), _ptr(b), _ptr(lg), _ptr(s)), "router")
    return lg, s


def select(scores, k):
    """Per row: (idx [T,k] int32, gates [T,k], gaps [T,k])."""
    s = _f64(np.atleast_2d(scores))
    T, E = s.shape
    idx = np.empty((T, k), np.int32)
    g = np.empty((T, k))
    gp = np.empty((T, k))
    for t in range(T):
        _check(_lib().oracle_select(_ptr(s[t]), E, k, _ptr(idx[t]), _ptr(g[t]), _ptr(gp[t])), "select")
    return idx, g, gp


def swiglu(x, wg, wu, wd):
    """One SwiGLU MLP on rows x ([T,H] float64)."""
    x = _f64(np.atleast_2d(x))
    wg, wu, wd = _u16(wg), _u16(wu), _u16(wd)
    H, I = wg.shape
    out = np.empty((x.shape[0], H))
    hbuf = np.empty(I)
    for t in range(x.shape[0]):
        _lib().oracle_swiglu(_ptr(x[t]), H, I, _ptr(wg), _ptr(wu), _ptr(wd), _ptr(out[t]), _ptr(hbuf))
    return out


def dense(x, wg, wu, wd, nthreads: int = 1):
    """A dense SwiGLU MLP layer on rows x ([T,H] float64): the same per-row computation as
    :func:`swiglu` (oracle_swiglu), with disjoint row ranges evaluated concurrently."""
    x = _f64(np.atleast_2d(x))
    wg, wu, wd = _u16(wg), _u16(wu), _u16(wd)
    H, I = wg.shape
    out = np.empty((x.shape[0], H))
    L = _lib()

    def run(a, b):
        hbuf = np.empty(I)
        for t in range(a, b):
            L.oracle_swiglu(_ptr(x[t]), H, I, _ptr(wg), _ptr(wu), _ptr(wd), _ptr(out[t]), _ptr(hbuf))

    parts = _split(x.shape[0], nthreads)
    if len(parts) <= 1:
        run(0, x.shape[0])
    else:
        with ThreadPoolExecutor(len(parts)) as ex:
            list(ex.map(lambda ab: run(*ab), parts))
    return out


def _split(T, nthreads):
    n = max(1, min(nthreads, T))
    b = np.linspace(0, T, n + 1).astype(int)
    return [(b[i], b[i + 1]) for i in range(n) if b[i + 1] > b[i]]


def forward(layer: Layer, x, nthreads: int = 1, want_scores: bool = False):
    """The layer on rows x ([T,H] float64).  Returns dict(y, idx, gates, gaps[, scores]).
    ``nthreads`` > 1 evaluates disjoint token ranges concurrently (each token's result is
    the same single-threaded computation)."""
    x = _f64(x)
    T = x.shape[0]
    k, E = layer.k, layer.E
    y = np.empty((T, layer.H))
    idx = np.empty((T, k), np.int32)
    g = np.empty((T, k))
    gp = np.empty((T, k))
    sc = np.empty((T, E)) if want_scores else None
    L = _lib()

    def run(a, b):
        if b <= a:
            return 0
        return L.oracle_moe_forward(ctypes.byref(layer._c), _ptr(x[a:b]), b - a, _ptr(y[a:b]),
                                    _ptr(idx[a:b]), _ptr(g[a:b]), _ptr(gp[a:b]),
                                    None if sc is None else _ptr(sc[a:b]))

    parts = _split(T, nthreads)
    if len(parts) <= 1:
        rcs = [run(0, T)]
    else:
        with ThreadPoolExecutor(len(parts)) as ex:
            rcs = list(ex.map(lambda ab: run(*ab), parts))
    for rc in rcs:
        _check(rc, "moe_forward")
    out = dict(y=y, idx=idx, gates=g, gaps=gp)
    if want_scores:
        out["scores"] = sc
    return out


def forward_given(layer: Layer, x, idx):
    """The layer on rows x with the chosen experts given (gates renormalised over them)."""
    x = _f64(x)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    y = np.empty((x.shape[0], layer.H))
    _check(_lib().oracle_moe_forward_given(ctypes.byref(layer._c), _ptr(x), x.shape[0], _ptr(idx), _ptr(y)),
           "moe_forward_given")
    return y


def permute(idx, E):
    """Stable counting sort of (token, slot) pairs by expert: counts, offsets, perm, inv."""
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    T, k = idx.shape
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    perm = np.empty(T * k, np.int32)
    inv = np.empty(T * k, np.int32)
    _check(_lib().oracle_permute(_ptr(idx), T, k, E, _ptr(counts), _ptr(offsets), _ptr(perm), _ptr(inv)),
           "permute")
    return counts, offsets, perm, inv


def rmsnorm(x, eps):
    x = _f64(x)
    r = np.empty_like(x)
    _lib().oracle_rmsnorm(_ptr(x), x.shape[0], x.shape[1], float(eps), _ptr(r))
    return r


def round_bf16(v) -> np.ndarray:
    """Elementwise rounding to the nearest bfloat16 value (ties to even), as float64."""
    L = _lib()
    a = _f64(v)
    return np.vectorize(L.oracle_round_bf16, otypes=[np.float64])(a) if a.size else a


def prenorm_input(x, eps):
    """The MoE input of a pre-norm layer: rmsnorm(x), handed to the layer as a bf16
    activation (rounded to bf16 like every tensor between the layer's steps)."""
    return round_bf16(rmsnorm(x, eps))


def prenorm_residual(layer: Layer, x, eps, nthreads: int = 1):
    """y = x + MoE(bf16(rmsnorm(x))); returns dict(y, idx, gates, gaps, r)."""
    x = _f64(x)
    r = prenorm_input(x, eps)
    out = forward(layer, r, nthreads=nthreads)
    out["y"] = x + out["y"]
    out["r"] = r
    return out


def swa_decode(q, k, v, sinks, pos, nthreads: int = 1):
    """Sliding-window decode attention with per-head sinks (oracle_swa_decode): q [B,nh,d],
    k, v [B,W,nkv,d] (bf16 bits, uint16), sinks [nh] fp32, pos [B] int32 -> out [B,nh,d]
    float64.  ``nthreads`` > 1 evaluates disjoint batch ranges concurrently."""
    q, k, v = _u16(q), _u16(k), _u16(v)
    sinks = np.ascontiguousarray(sinks, dtype=np.float32)
    pos = np.ascontiguousarray(pos, dtype=np.int32)
    B, nh, d = q.shape
    W, nkv = k.shape[1], k.shape[2]
    out = np.empty((B, nh, d))
    L = _lib()

    def run(a, b):
        if b <= a:
            return 0
        return L.oracle_swa_decode(_ptr(q[a:b]), _ptr(k[a:b]), _ptr(v[a:b]), _ptr(sinks), _ptr(pos[a:b]), b - a, nh,
                                   nkv, d, W, _ptr(out[a:b]))

    parts = _split(B, nthreads)
    if len(parts) <= 1:
        rcs = [run(0, B)]
    else:
        with ThreadPoolExecutor(len(parts)) as ex:
            rcs = list(ex.map(lambda ab: run(*ab), parts))
    for rc in rcs:
        _check(rc, "swa_decode")
    return out


def e2m1_to_f64(code: int) -> float:
    return _lib().oracle_e2m1_to_f64(int(code))


def e4m3_to_f64(byte: int) -> float:
    return _lib().oracle_e4m3_to_f64(int(byte))


def nvfp4_dequant(codes, scales, tensor_scale) -> np.ndarray:
    """W [K, N] float64 from the K-major NVFP4 encoding: codes [N, K/2] (uint8, two consecutive k
    per byte, the lower k in the low nibble), E4M3 block scales [N, K/16] (uint8) and the fp32
    tensor scale."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    N, K = codes.shape[0], codes.shape[1] * 2
    out = np.empty((K, N))
    _check(_lib().oracle_nvfp4_dequant(_ptr(codes), _ptr(scales), float(tensor_scale), K, N, _ptr(out)),
           "nvfp4_dequant")
    return out


def f64_to_bf16_exact(w) -> np.ndarray:
    """bf16 bit patterns of float64 values that bf16 holds exactly (raises otherwise): NVFP4
    weights with a power-of-two tensor scale are such values (a 2-bit by 4-bit significand
    product), so the bf16 layer above computes the dequantised layer exactly."""
    w = np.asarray(w, dtype=np.float64)
    f = w.astype(np.float32)
    if not np.array_equal(f.astype(np.float64), w):
        raise ValueError("not representable in float32")
    bits = f.view(np.uint32)
    if np.any(bits & np.uint32(0xFFFF)):
        raise ValueError("not representable in bf16")
    return (bits >> np.uint32(16)).astype(np.uint16)
