"""Seeded synthetic inputs for the MoE FFN layer and the Gated DeltaNet scan (data only: none
of their arithmetic).

The generator itself (splitmix64 words, 12-term Irwin-Hall values, bf16 rounding) is C in
synth_host.c / synth_dev.cu; its definition is in synth.h.  This module composes streams
into the tensors of one layer.  The same functions feed the oracle (host arrays) and the
CUDA library (device fills), so both sides receive identical bits.

Layouts (row-major, bf16 as uint16 bits; every weight is stored output-major, the input
dimension contiguous, like a linear layer's weight matrix):
  x      [T][d]          sigma 1
  w_r    [E][d]          sigma 0.05   (the router; mathematically the d x E matrix W_r)
  w_gate [E][f][d]       sigma 0.02
  w_up   [E][f][d]       sigma 0.02
  w_down [E][d][f]       sigma 0.02
  ws_gate, ws_up [fs][d], ws_down [d][fs]   sigma 0.02 (the shared expert)
Element (r, c) of a tensor is element r*cols + c of its stream, so any expert or row range
can be produced on its own.

4-bit group-affine experts (the same names, one group per 64 inputs of a row): codes
[rows][K/2] uint8 (two codes per byte, the lower nibble first), scales and biases
[rows][K/64] bf16, with K the row length (d for gate/up, f or fs for down); the dequantized
weight is scale*q + bias (see synth.h for how they are drawn).
"""
import ctypes
import os
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_lib = None

# tensor ids inside a stream id
X, W_R, W_GATE, W_UP, W_DOWN, WS_GATE, WS_UP, WS_DOWN, RANKS = range(1, 10)

SIGMA_X = 1.0
SIGMA_ROUTER = 0.05
SIGMA_EXPERT = 0.02


def stream_id(tensor, layer=0, rnd=0):
    """64-bit stream id of (tensor, layer, redraw round)."""
    return (int(tensor) << 40) | (int(layer) << 20) | int(rnd)


def lib():
    global _lib
    if _lib is None:
        path = os.path.join(_HERE, "libsynth.so")
        if not os.path.exists(path):
            from . import build as _b
            _b.build()
        L = ctypes.CDLL(path)
        L.synth_key.restype = ctypes.c_uint64
        L.synth_key.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
        L.synth_word.restype = ctypes.c_uint64
        L.synth_word.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
        L.synth_normal_bf16.restype = None
        L.synth_normal_bf16.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                                        ctypes.c_uint64, ctypes.c_float, ctypes.c_void_p,
                                        ctypes.c_int]
        L.synth_permutation.restype = None
        L.synth_permutation.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int32,
                                        ctypes.c_void_p]
        L.synth_bytes.restype = None
        L.synth_bytes.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                                  ctypes.c_uint64, ctypes.c_void_p]
        L.synth_q4_affine.restype = None
        L.synth_q4_affine.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                                      ctypes.c_uint64, ctypes.c_float, ctypes.c_void_p,
                                      ctypes.c_void_p]
        L.synth_bytes_device.restype = ctypes.c_int
        L.synth_bytes_device.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                                         ctypes.c_uint64, ctypes.c_void_p, ctypes.c_void_p]
        L.synth_q4_affine_device.restype = ctypes.c_int
        L.synth_q4_affine_device.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                                             ctypes.c_uint64, ctypes.c_float, ctypes.c_void_p,
                                             ctypes.c_void_p, ctypes.c_void_p]
        L.synth_uniform_f32.restype = None
        L.synth_uniform_f32.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                                        ctypes.c_uint64, ctypes.c_float, ctypes.c_float,
                                        ctypes.c_void_p]
        L.synth_uniform_f32_device.restype = ctypes.c_int
        L.synth_uniform_f32_device.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                                               ctypes.c_uint64, ctypes.c_float, ctypes.c_float,
                                               ctypes.c_void_p, ctypes.c_void_p]
        L.synth_normal_bf16_device.restype = ctypes.c_int
        L.synth_normal_bf16_device.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                                               ctypes.c_uint64, ctypes.c_float, ctypes.c_void_p,
                                               ctypes.c_void_p]
        _lib = L
    return _lib


def host_threads():
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return os.cpu_count() or 1


def normal_bf16(seed, stream, offset, n, sigma, nthreads=None):
    out = np.empty(int(n), dtype=np.uint16)
    if n:
        lib().synth_normal_bf16(seed, stream, offset, n, sigma, out.ctypes.data,
                                host_threads() if nthreads is None else nthreads)
    return out


def normal_bf16_device(seed, stream, offset, n, sigma, dev_ptr, cuda_stream=0):
    rc = lib().synth_normal_bf16_device(seed, stream, offset, n, sigma, dev_ptr, cuda_stream)
    if rc != 0:
        raise RuntimeError(f"synth device fill failed: cudaError {rc}")


def permutation(seed, stream, n):
    out = np.empty(int(n), dtype=np.int32)
    lib().synth_permutation(seed, stream, n, out.ctypes.data)
    return out


@dataclass(frozen=True)
class Dims:
    """Shape of one MoE layer: d hidden, E experts, k kept per token, f expert inner dim,
    fs shared-expert inner dim."""
    d: int
    E: int = 256
    k: int = 8
    f: int = 512
    fs: int = 512


# tensor name -> (tensor id, shape function, sigma)
_SPEC = {
    "w_r": (W_R, lambda D: (D.E, D.d), SIGMA_ROUTER),
    "w_gate": (W_GATE, lambda D: (D.E, D.f, D.d), SIGMA_EXPERT),
    "w_up": (W_UP, lambda D: (D.E, D.f, D.d), SIGMA_EXPERT),
    "w_down": (W_DOWN, lambda D: (D.E, D.d, D.f), SIGMA_EXPERT),
    "ws_gate": (WS_GATE, lambda D: (D.fs, D.d), SIGMA_EXPERT),
    "ws_up": (WS_UP, lambda D: (D.fs, D.d), SIGMA_EXPERT),
    "ws_down": (WS_DOWN, lambda D: (D.d, D.fs), SIGMA_EXPERT),
}
WEIGHT_NAMES = tuple(_SPEC)


def weight_shape(name, dims):
    return _SPEC[name][1](dims)


def host_weight(seed, layer, name, dims, expert=None):
    """Whole tensor `name` of `layer`, or only expert `expert`'s slice of a routed tensor."""
    tid, shp, sigma = _SPEC[name]
    shape = shp(dims)
    if expert is None:
        n = int(np.prod(shape))
        return normal_bf16(seed, stream_id(tid, layer), 0, n, sigma).reshape(shape)
    per = int(np.prod(shape[1:]))
    return normal_bf16(seed, stream_id(tid, layer), int(expert) * per, per,
                       sigma).reshape(shape[1:])


def device_weight(seed, layer, name, dims, dev_ptr, cuda_stream=0):
    tid, shp, sigma = _SPEC[name]
    n = int(np.prod(shp(dims)))
    normal_bf16_device(seed, stream_id(tid, layer), 0, n, sigma, dev_ptr, cuda_stream)


def x_rows(seed, layer, T, d, rounds=None):
    """x [T][d]; row t is drawn from redraw round rounds[t] (default 0 for every row)."""
    if rounds is None:
        return normal_bf16(seed, stream_id(X, layer, 0), 0, T * d, SIGMA_X).reshape(T, d)
    rounds = np.asarray(rounds, dtype=np.int64)
    x = np.empty((T, d), dtype=np.uint16)
    for r in np.unique(rounds):
        rows = np.nonzero(rounds == r)[0]
        if r == 0:
            full = normal_bf16(seed, stream_id(X, layer, 0), 0, T * d, SIGMA_X).reshape(T, d)
            x[rows] = full[rows]
            continue
        for t in rows:
            x[t] = normal_bf16(seed, stream_id(X, layer, int(r)), int(t) * d, d, SIGMA_X)
    return x


def skew_bias(seed, layer, E):
    """Zipf-like per-expert router bias b_e = 2*log(1/rank_e^1.2) = -2.4*ln(rank_e), ranks
    1..E taken from a seeded random permutation of the experts (fp32)."""
    perm = permutation(seed, stream_id(RANKS, layer), E)
    rank = np.empty(E, dtype=np.float64)
    rank[perm] = np.arange(1, E + 1, dtype=np.float64)
    return (-2.4 * np.log(rank)).astype(np.float32)


# 4-bit weights: stream ids of the codes and of the scales/biases of tensor t
Q4_CODES, Q4_AFFINE = 16, 32
Q4_GROUP = 64
Q4_BASE = 0.02 / 4.61  # spread of s*(q - 8), q uniform on 0..15: 4.61 s
Q4_NAMES = tuple(n for n in WEIGHT_NAMES if n != "w_r")


def q4_shapes(name, dims):
    """(codes shape, scales/biases shape) of 4-bit tensor `name`."""
    shape = weight_shape(name, dims)
    K = shape[-1]
    return shape[:-1] + (K // 2,), shape[:-1] + (K // Q4_GROUP,)


def q4_host(seed, layer, name, dims, expert=None):
    """(codes uint8, scales bf16 bits, biases bf16 bits) of 4-bit tensor `name` of `layer`,
    or only expert `expert`'s slice of a routed tensor."""
    tid = _SPEC[name][0]
    cs, gs = q4_shapes(name, dims)
    if expert is not None:
        cs, gs = cs[1:], gs[1:]
    nc, ng = int(np.prod(cs)), int(np.prod(gs))
    oc = 0 if expert is None else int(expert) * nc
    og = 0 if expert is None else int(expert) * ng
    codes = np.empty(nc, dtype=np.uint8)
    scales = np.empty(ng, dtype=np.uint16)
    biases = np.empty(ng, dtype=np.uint16)
    lib().synth_bytes(seed, stream_id(Q4_CODES + tid, layer), oc, nc, codes.ctypes.data)
    lib().synth_q4_affine(seed, stream_id(Q4_AFFINE + tid, layer), og, ng, Q4_BASE,
                          scales.ctypes.data, biases.ctypes.data)
    return codes.reshape(cs), scales.reshape(gs), biases.reshape(gs)


def q4_device(seed, layer, name, dims, codes_ptr, scales_ptr, biases_ptr, cuda_stream=0):
    """Device fill of the whole 4-bit tensor `name` (the bits of q4_host)."""
    tid = _SPEC[name][0]
    cs, gs = q4_shapes(name, dims)
    rc = lib().synth_bytes_device(seed, stream_id(Q4_CODES + tid, layer), 0, int(np.prod(cs)),
                                  codes_ptr, cuda_stream)
    if rc == 0:
        rc = lib().synth_q4_affine_device(seed, stream_id(Q4_AFFINE + tid, layer), 0,
                                          int(np.prod(gs)), Q4_BASE, scales_ptr, biases_ptr,
                                          cuda_stream)
    if rc != 0:
        raise RuntimeError(f"synth device fill failed: cudaError {rc}")


def uniform_f32(seed, stream, offset, n, lo, hi):
    out = np.empty(int(n), dtype=np.float32)
    if n:
        lib().synth_uniform_f32(seed, stream, offset, n, lo, hi, out.ctypes.data)
    return out


def uniform_f32_device(seed, stream, offset, n, lo, hi, dev_ptr, cuda_stream=0):
    rc = lib().synth_uniform_f32_device(seed, stream, offset, n, lo, hi, dev_ptr, cuda_stream)
    if rc != 0:
        raise RuntimeError(f"synth device fill failed: cudaError {rc}")


# ---- inputs of the Gated DeltaNet recurrent scan (one layer, H heads)
#
#   q, k   [T][H][dk]   bf16, sigma dk^-1/2 (so that |k|^2 is close to 1, the regime in which the
#                       delta rule's update I - beta k k^T is a contraction for beta in [0, 1))
#   v      [T][H][dv]   bf16, sigma 1
#   alpha  [T][H]       fp32 uniform on [0.80, 1.00): the per-token decay gate
#   beta   [T][H]       fp32 uniform on [0, 1): the per-token write strength
#   s0     [H][dk][dv]  fp32 holding bf16 values of sigma 0.25 (the state a previous prompt chunk
#                       leaves), or zeros (the first chunk)
# Element (t, h, i) of q is element (t H + h) dk + i of its stream, so a range of tokens can be
# produced on its own.
GDN_Q, GDN_K, GDN_V, GDN_ALPHA, GDN_BETA, GDN_S0 = range(40, 46)
GDN_ALPHA_RANGE = (0.80, 1.0)
GDN_BETA_RANGE = (0.0, 1.0)
SIGMA_GDN_V = 1.0
SIGMA_GDN_S0 = 0.25


def gdn_sigma_qk(dk):
    return float(np.float32(1.0 / np.sqrt(dk)))


def gdn_inputs(seed, T, H, dk, dv, layer=0, t0=0, zero_state=False):
    """Host inputs (q, k, v as bf16 bits; alpha, beta, s0 fp32) of tokens t0 .. t0 + T - 1."""
    sq = gdn_sigma_qk(dk)
    q = normal_bf16(seed, stream_id(GDN_Q, layer), t0 * H * dk, T * H * dk, sq).reshape(T, H, dk)
    k = normal_bf16(seed, stream_id(GDN_K, layer), t0 * H * dk, T * H * dk, sq).reshape(T, H, dk)
    v = normal_bf16(seed, stream_id(GDN_V, layer), t0 * H * dv, T * H * dv,
                    SIGMA_GDN_V).reshape(T, H, dv)
    alpha = uniform_f32(seed, stream_id(GDN_ALPHA, layer), t0 * H, T * H,
                        *GDN_ALPHA_RANGE).reshape(T, H)
    beta = uniform_f32(seed, stream_id(GDN_BETA, layer), t0 * H, T * H,
                       *GDN_BETA_RANGE).reshape(T, H)
    if zero_state:
        s0 = np.zeros((H, dk, dv), dtype=np.float32)
    else:
        s0 = bf16_to_f32(normal_bf16(seed, stream_id(GDN_S0, layer), 0, H * dk * dv,
                                     SIGMA_GDN_S0)).reshape(H, dk, dv)
    return q, k, v, alpha, beta, s0


def gdn_inputs_device(seed, T, H, dk, dv, q_ptr, k_ptr, v_ptr, alpha_ptr, beta_ptr,
                      s0_bf16_ptr=None, layer=0, cuda_stream=0):
    """Device fills of the same bits as gdn_inputs (t0 = 0).  s0 is filled as bf16 bits; the
    caller widens it to fp32 (exact) or passes zeros."""
    sq = gdn_sigma_qk(dk)
    normal_bf16_device(seed, stream_id(GDN_Q, layer), 0, T * H * dk, sq, q_ptr, cuda_stream)
    normal_bf16_device(seed, stream_id(GDN_K, layer), 0, T * H * dk, sq, k_ptr, cuda_stream)
    normal_bf16_device(seed, stream_id(GDN_V, layer), 0, T * H * dv, SIGMA_GDN_V, v_ptr,
                       cuda_stream)
    uniform_f32_device(seed, stream_id(GDN_ALPHA, layer), 0, T * H, *GDN_ALPHA_RANGE, alpha_ptr,
                       cuda_stream)
    uniform_f32_device(seed, stream_id(GDN_BETA, layer), 0, T * H, *GDN_BETA_RANGE, beta_ptr,
                       cuda_stream)
    if s0_bf16_ptr is not None:
        normal_bf16_device(seed, stream_id(GDN_S0, layer), 0, H * dk * dv, SIGMA_GDN_S0,
                           s0_bf16_ptr, cuda_stream)


def bf16_to_f32(a):
    """Widen bf16 bits (uint16) to float32 exactly."""
    return (np.asarray(a, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16(a):
    """Round float32 to bf16 bits (round to nearest even; finite inputs)."""
    u = np.asarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


__all__ = ["Dims", "stream_id", "normal_bf16", "normal_bf16_device", "permutation",
           "host_weight", "device_weight", "x_rows", "skew_bias", "bf16_to_f32", "f32_to_bf16",
           "weight_shape", "WEIGHT_NAMES", "q4_shapes", "q4_host", "q4_device", "Q4_NAMES",
           "uniform_f32", "uniform_f32_device", "gdn_inputs", "gdn_inputs_device"]
