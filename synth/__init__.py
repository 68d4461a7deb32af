"""Seeded synthetic inputs for the Flint-shaped MoE layer.

This module is shared by the fp64 oracle side (tests, CPU baseline) and the CUDA
side (tests, bench).  It holds no arithmetic of the MoE method itself: it only
draws numbers.  Every value is a pure function of (seed, tag, element index), so
any slice of any tensor can be regenerated without generating the rest, and the
device twin (``synth/gen.cu``) produces bit-identical arrays on the GPU.

Generator (the same on host and device):

* stream: splitmix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014).  The per-tensor state is
  ``key = mix64(mix64(seed + GOLDEN) ^ (tag * TAGMUL))``; element ``i`` consumes
  outputs ``2i+1`` and ``2i+2`` of the stream started at ``key``, i.e.
  ``z_j = mix64(key + j * GOLDEN)`` (all arithmetic mod 2**64).
* normal deviate: Box--Muller (Box and Muller, 1958),
  ``u1 = ((z1 >> 11) + 1) * 2**-53`` in (0, 1], ``u2 = (z2 >> 11) * 2**-53`` in
  [0, 1), ``n = sqrt(-2 ln u1) * cos(2*pi*u2)`` in float64.
* value: ``float32(sigma * n)`` (round to nearest), then bfloat16 by
  round-to-nearest-even on the float32 bits.

Host and device use different libm ``log``/``cos``; a last-bit difference in
float64 changes the bf16 result only when it straddles a rounding boundary, a
chance of order 2**-45 per element.
"""
from __future__ import annotations

import ctypes
import math
import os

import numpy as np

GOLDEN = 0x9E3779B97F4A7C15
TAGMUL = 0xD1B54A32D192ED03
M1 = 0xBF58476D1CE4E5B9
M2 = 0x94D049BB133111EB
TWO_PI = 6.283185307179586  # the float64 nearest to 2*pi, used verbatim on both sides

# Tensor tags.  The layer index of a stacked model is folded into the seed.
TAG_X = 1
TAG_ROUTER = 2
TAG_BIAS = 3
TAG_GATE = 4
TAG_UP = 5
TAG_DOWN = 6
TAG_SGATE = 7
TAG_SUP = 8
TAG_SDOWN = 9
TAG_PERM = 10
TAG_DGATE = 11  # dense MLP layers
TAG_DUP = 12
TAG_DDOWN = 13
TAG_Q = 14  # sliding-window decode attention
TAG_K = 15
TAG_V = 16
TAG_SINK = 17

_MASK = (1 << 64) - 1


def mix64_int(z: int) -> int:
    """splitmix64 output function on a Python int (reference scalar form)."""
    z &= _MASK
    z = ((z ^ (z >> 30)) * M1) & _MASK
    z = ((z ^ (z >> 27)) * M2) & _MASK
    return z ^ (z >> 31)


def tensor_key(seed: int, tag: int) -> int:
    return mix64_int(mix64_int((seed + GOLDEN) & _MASK) ^ ((tag * TAGMUL) & _MASK))


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * np.uint64(M1)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(M2)
    return z ^ (z >> np.uint64(31))


def f32_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bits, round to nearest even (inputs are finite)."""
    b = np.ascontiguousarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))
    return (b >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16_at(seed: int, tag: int, idx, sigma: float) -> np.ndarray:
    """bf16 bits of elements ``idx`` (any int array) of tensor (seed, tag)."""
    with np.errstate(over="ignore"):
        idx = np.asarray(idx, dtype=np.uint64)
        key = np.uint64(tensor_key(seed, tag))
        g = np.uint64(GOLDEN)
        z1 = _mix64(key + (np.uint64(2) * idx + np.uint64(1)) * g)
        z2 = _mix64(key + (np.uint64(2) * idx + np.uint64(2)) * g)
    u1 = ((z1 >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)
    u2 = (z2 >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    n = np.sqrt(-2.0 * np.log(u1)) * np.cos(TWO_PI * u2)
    return f32_to_bf16_bits((float(sigma) * n).astype(np.float32))


def normal_bf16(seed: int, tag: int, n: int, sigma: float, start: int = 0,
                chunk: int = 1 << 22) -> np.ndarray:
    """bf16 bits of elements [start, start+n) of tensor (seed, tag)."""
    out = np.empty(n, dtype=np.uint16)
    for c0 in range(0, n, chunk):
        c1 = min(n, c0 + chunk)
        out[c0:c1] = normal_bf16_at(seed, tag, np.arange(start + c0, start + c1, dtype=np.uint64), sigma)
    return out


def permutation(seed: int, n: int) -> np.ndarray:
    """A seeded permutation of range(n): argsort of splitmix64 draws (ties by index)."""
    with np.errstate(over="ignore"):
        key = np.uint64(tensor_key(seed, TAG_PERM))
        z = _mix64(key + (np.arange(n, dtype=np.uint64) + np.uint64(1)) * np.uint64(GOLDEN))
    return np.argsort(z, kind="stable").astype(np.int64)


# --------------------------------------------------------------------------------------
# Device twin (synth/gen.cu -> synth/libsynth.so).  Only data generation lives there.

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = None


def lib_path() -> str:
    return os.path.join(_HERE, "libsynth.so")


def build(verbose: bool = False) -> str:
    import subprocess
    src = os.path.join(_HERE, "gen.cu")
    out = lib_path()
    cmd = ["nvcc", "-O3", "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo",
           "-Xcompiler", "-fPIC", "-shared", "-o", out, src]
    if verbose:
        print(" ".join(cmd))
    subprocess.check_call(cmd)
    return out


def _lib():
    global _LIB
    if _LIB is None:
        path = lib_path()
        if not os.path.exists(path):
            raise RuntimeError(f"synth device generator not built: {path} (run __graft_entry__.build())")
        _LIB = ctypes.CDLL(path)
        _LIB.synth_normal_bf16.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint64,
                                           ctypes.c_uint64, ctypes.c_uint32, ctypes.c_double,
                                           ctypes.c_void_p]
        _LIB.synth_normal_bf16.restype = ctypes.c_int
    return _LIB


def device_normal_bf16(dst_ptr: int, n: int, seed: int, tag: int, sigma: float,
                       start: int = 0, stream: int = 0) -> None:
    """Fill ``n`` bf16 values at device pointer ``dst_ptr`` with elements
    [start, start+n) of tensor (seed, tag); bit-identical to :func:`normal_bf16`."""
    rc = _lib().synth_normal_bf16(ctypes.c_void_p(dst_ptr), n, start, seed & _MASK, tag,
                                  float(sigma), ctypes.c_void_p(stream))
    if rc != 0:
        raise RuntimeError(f"synth_normal_bf16 failed with CUDA error {rc}")


def torch_normal_bf16(shape, seed: int, tag: int, sigma: float, device="cuda", start: int = 0):
    """A torch bf16 tensor of ``shape`` filled by the generator (device or host)."""
    import torch
    n = int(np.prod(shape))
    if str(device).startswith("cuda"):
        t = torch.empty(shape, dtype=torch.bfloat16, device=device)
        if n:
            device_normal_bf16(t.data_ptr(), n, seed, tag, sigma, start,
                               torch.cuda.current_stream(t.device).cuda_stream)
        return t
    bits = normal_bf16(seed, tag, n, sigma, start)
    return torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).reshape(shape)


SIGMA_X = 1.0
SIGMA_ROUTER = 1.0 / math.sqrt(2048.0)
SIGMA_EXPERT = 0.02
SIGMA_BIAS = math.sqrt(0.5)


# --------------------------------------------------------------------------------------
# Flint-layer input sets (weights and token rows), as used by the tests and the benchmark.

LAYER_SHAPES = {
    "w_router": (2048, 256),
    "w_gate": (256, 2048, 512),
    "w_up": (256, 2048, 512),
    "w_down": (256, 512, 2048),
    "ws_gate": (2048, 1024),
    "ws_up": (2048, 1024),
    "ws_down": (1024, 2048),
}
_LAYER_TAGS = {"w_router": (TAG_ROUTER, SIGMA_ROUTER), "w_gate": (TAG_GATE, SIGMA_EXPERT),
               "w_up": (TAG_UP, SIGMA_EXPERT), "w_down": (TAG_DOWN, SIGMA_EXPERT),
               "ws_gate": (TAG_SGATE, SIGMA_EXPERT), "ws_up": (TAG_SUP, SIGMA_EXPERT),
               "ws_down": (TAG_SDOWN, SIGMA_EXPERT)}


def flint_weights(seed: int, device="cuda", bias: str | None = None, bias_seed: int | None = None):
    """One layer's weights, generated on ``device``: router ~N(0, 1/2048), expert and shared
    matrices ~N(0, 0.02^2), all bf16.  ``bias``: None (no router bias), "normal" (fp32
    bf16-valued ~N(0, 0.5), seed ``bias_seed``) or "adversarial" (see
    :func:`adversarial_bias_and_router`)."""
    import torch
    w = {}
    for name, shape in LAYER_SHAPES.items():
        tag, sigma = _LAYER_TAGS[name]
        w[name] = torch_normal_bf16(shape, seed, tag, sigma, device=device)
    w["router_bias"] = None
    if bias == "normal":
        b = torch_normal_bf16((256,), seed if bias_seed is None else bias_seed, TAG_BIAS, SIGMA_BIAS, device=device)
        w["router_bias"] = b.float().contiguous()
    elif bias == "adversarial":
        hot, cold, neutral = adversarial_sets(5 if bias_seed is None else bias_seed)
        b = torch.zeros(256, dtype=torch.float32)
        b[hot] = 8.0
        b[cold] = -8.0
        w["router_bias"] = b.to(device)
        wr = w["w_router"]
        # exact score ties: duplicated router columns with equal bias
        wr[:, hot[1]] = wr[:, hot[0]]
        wr[:, hot[3]] = wr[:, hot[2]]
        wr[:, neutral[1]] = wr[:, neutral[0]]
    elif bias is not None:
        raise ValueError(bias)
    return w


DENSE_SHAPES = {"w_gate": (2048, 6144), "w_up": (2048, 6144), "w_down": (6144, 2048)}
_DENSE_TAGS = {"w_gate": TAG_DGATE, "w_up": TAG_DUP, "w_down": TAG_DDOWN}


def dense_weights(seed: int, device="cuda"):
    """A dense SwiGLU MLP layer's weights (width 6144), bf16 ~N(0, 0.02^2) like the experts'."""
    return {name: torch_normal_bf16(shape, seed, _DENSE_TAGS[name], SIGMA_EXPERT, device=device)
            for name, shape in DENSE_SHAPES.items()}


def adversarial_sets(seed: int = 5):
    """A seeded permutation of the 256 experts split into 8 hot, 200 cold, 48 neutral."""
    pi = permutation(seed, 256)
    return [int(v) for v in pi[:8]], [int(v) for v in pi[8:208]], [int(v) for v in pi[208:]]


def weights_to_host(w, experts=None):
    """uint16 numpy copies of a layer's weights (only ``experts`` of the routed ones, as a
    dict, when given), plus the fp32 bias or None."""
    out = {}
    for name in ("w_router", "ws_gate", "ws_up", "ws_down"):
        out[name] = w[name].contiguous().view(__import__("torch").int16).cpu().numpy().view(np.uint16)
    for name in ("w_gate", "w_up", "w_down"):
        t = w[name]
        if experts is None:
            out[name] = t.contiguous().view(__import__("torch").int16).cpu().numpy().view(np.uint16)
        else:
            out[name] = {int(e): t[int(e)].contiguous().view(__import__("torch").int16).cpu().numpy().view(np.uint16)
                         for e in experts}
    b = w.get("router_bias")
    out["router_bias"] = None if b is None else b.detach().float().cpu().numpy()
    return out


# --------------------------------------------------------------------------------------
# Sliding-window decode attention inputs: 32 query heads, 4 KV heads, head dimension 128, a ring
# of 513 cached tokens per sequence.  q and k rows ~N(0, 1) (what a per-head RMSNorm leaves),
# v ~N(0, 1), one sink logit per head ~N(0, 1) (bf16-valued fp32), and a length mix: the current
# token's position cycles through SWA_POSITIONS, so some sequences are shorter than the window
# (0, 17, 511 tokens back) and the rest fill it.
SWA_HEADS, SWA_KV_HEADS, SWA_HEAD_DIM, SWA_WINDOW = 32, 4, 128, 513
SWA_POSITIONS = (4095, 511, 0, 512, 131071, 17, 513, 1023)


def swa_inputs(B: int, seed: int, device="cuda"):
    """dict(q [B,32,128], k, v [B,513,4,128] bf16, sinks [32] fp32, pos [B] int32)."""
    import torch
    q = torch_normal_bf16((B, SWA_HEADS, SWA_HEAD_DIM), seed, TAG_Q, 1.0, device=device)
    k = torch_normal_bf16((B, SWA_WINDOW, SWA_KV_HEADS, SWA_HEAD_DIM), seed, TAG_K, 1.0, device=device)
    v = torch_normal_bf16((B, SWA_WINDOW, SWA_KV_HEADS, SWA_HEAD_DIM), seed, TAG_V, 1.0, device=device)
    sinks = torch_normal_bf16((SWA_HEADS,), seed, TAG_SINK, 1.0, device=device).float().contiguous()
    pos = torch.tensor([SWA_POSITIONS[b % len(SWA_POSITIONS)] for b in range(B)], dtype=torch.int32, device=device)
    return dict(q=q, k=k, v=v, sinks=sinks, pos=pos)


# --------------------------------------------------------------------------------------
# NVFP4 expert weights.  The layer consumes NVFP4 weights as given; this module prepares seeded
# synthetic ones by quantising the seeded bf16 weights above (input preparation, done once):
#   tensor scale  t = 2^ceil(log2(amax / (6 * 448)))  (a power of two, one per matrix)
#   block scale   s = the smallest E4M3 value >= amax(block of 16 along K) / 6 / t
#   code          e2m1 = round(w / (s t)) to the nearest of 0, .5, 1, 1.5, 2, 3, 4, 6, ties to the
#                 even code, sign kept
# Layouts (K-major, for W [K][N] of y = x W): codes [.., N, K/2] uint8 (W[2j][n] in the low
# nibble of byte (n, j), W[2j+1][n] in the high), scales [.., N, K/16] uint8 (E4M3 bits), tensor
# scales [..] fp32.

_E2M1_MID = (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)  # midpoints between the magnitudes


def _e2m1_round_code(a):
    """Magnitude code 0..7 of |v| (torch float32 tensor a >= 0), nearest with ties to even."""
    import torch
    mids = torch.tensor(_E2M1_MID, dtype=torch.float32, device=a.device)
    idx = torch.bucketize(a, mids, right=False)  # a <= mids[i] -> i (a tie goes to the lower code)
    # a tie at mids[i] goes to the even code of the pair (i, i + 1)
    tie = torch.zeros_like(a, dtype=torch.bool)
    for i, m in enumerate(_E2M1_MID):
        tie |= (a == m) & torch.tensor(i % 2 == 1, device=a.device)
    return torch.where(tie, idx + 1, idx).clamp(max=7)


def nvfp4_quantize(w):
    """(codes, scales, tensor_scale) of bf16 matrices w [..., K, N] (torch; any device)."""
    import torch
    lead = w.shape[:-2]
    K, N = w.shape[-2], w.shape[-1]
    w32 = w.float().reshape(-1, K, N)
    M = w32.shape[0]
    amax = w32.abs().amax(dim=(1, 2))
    ts = torch.where(amax > 0, torch.exp2(torch.ceil(torch.log2(amax / (6.0 * 448.0)))), torch.ones_like(amax))
    blk = w32.view(M, K // 16, 16, N)
    need = blk.abs().amax(dim=2) / 6.0 / ts.view(M, 1, 1)  # the block scale must reach this
    sb = need.to(torch.float8_e4m3fn)
    bits = sb.view(torch.uint8)
    low = sb.float() < need
    bits = torch.where(low, bits + 1, bits)  # round up to the next E4M3 value
    sbf = bits.view(torch.float8_e4m3fn).float()
    denom = (sbf * ts.view(M, 1, 1)).unsqueeze(2)  # [M, K/16, 1, N]
    v = torch.where(denom > 0, blk / torch.where(denom > 0, denom, torch.ones_like(denom)), torch.zeros_like(blk))
    mag = _e2m1_round_code(v.abs())
    code = (mag | torch.where(v < 0, 8, 0)).to(torch.uint8).view(M, K, N)
    code = torch.where(mag.view(M, K, N) == 0, torch.zeros_like(code), code)  # no negative zero
    code = code.transpose(1, 2)  # [M, N, K]: K-major
    packed = (code[..., 0::2] | (code[..., 1::2] << 4)).contiguous()
    return (packed.view(*lead, N, K // 2), bits.transpose(1, 2).contiguous().view(*lead, N, K // 16),
            ts.view(*lead) if lead else ts.view(()))


def nvfp4_weights(w):
    """NVFP4 copies of a layer's expert matrices (routed and shared; the router stays bf16):
    dict name -> (codes, scales, tensor_scale), quantised in chunks of experts on w's device."""
    import torch
    out = {}
    for name in ("w_gate", "w_up", "w_down"):
        parts = [nvfp4_quantize(w[name][e0:e0 + 32]) for e0 in range(0, w[name].shape[0], 32)]
        out[name] = tuple(torch.cat([p[i] for p in parts]) for i in range(3))
    for name in ("ws_gate", "ws_up", "ws_down"):
        out[name] = nvfp4_quantize(w[name])
    return out
