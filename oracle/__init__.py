"""CPU oracles of the MoE FFN layer and of the Gated DeltaNet recurrent scan -- TEST
INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the CPU-baseline timing leg of the benchmark use this
package; the product library and its Python binding never import it.  The arithmetic lives in
moe_oracle.cpp (plain loops, fp32 over bf16 inputs) and gdn_oracle.cpp (the scan, fp64); this
module marshals numpy arrays and
implements the input-drawing rule that keeps routing decisions well separated:

  a token is kept only if the gap between its k-th and (k+1)-th largest router logit,
  computed in fp64 from the exact bf16 inputs, is at least 1e-3; otherwise its x row is
  redrawn from the next redraw round of the same stream until it passes.

Parity status of each function is pinned by tests/test_oracle_pins.py.
"""
import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_lib = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I = ctypes.c_int


class _Dims(ctypes.Structure):
    _fields_ = [("d", _I), ("E", _I), ("k", _I), ("f", _I), ("fs", _I)]


class _Q4(ctypes.Structure):
    _fields_ = [("codes", _P), ("scales", _P), ("biases", _P)]


def lib():
    global _lib
    if _lib is None:
        # ORACLE_LIB lets the mutation test load a deliberately broken copy of the oracle
        path = os.environ.get("ORACLE_LIB") or os.path.join(_HERE, "liboracle.so")
        if not os.path.exists(path):
            from . import build as _b
            _b.build()
        L = ctypes.CDLL(path)
        L.oracle_router_logits_f64.argtypes = [_P, _I64, _I, _P, _I, _P, _P, _I]
        L.oracle_router_logits_f32.argtypes = [_P, _I64, _I, _P, _I, _P, _P, _I]
        L.oracle_select.argtypes = [_P, _I64, _I, _I, _P, _P]
        L.oracle_route_structure.argtypes = [_P, _I64, _I, _I, _P, _P, _P, _P]
        L.oracle_expert_ffn.argtypes = [_P, _I, _P, _P, _P, _I, _P, _P]
        L.oracle_forward.argtypes = [ctypes.POINTER(_Dims), _P, _I64, _P, _P, _P, _P, _P, _P, _P,
                                     _P, _P, _I64, _P, _P, _P, _I]
        L.oracle_dequant_q4.argtypes = [ctypes.POINTER(_Q4), _I64, _I, _P]
        L.oracle_forward_q4.argtypes = [ctypes.POINTER(_Dims), _P, _I64, _P, _P, _P, _P, _P,
                                        ctypes.POINTER(_Q4), ctypes.POINTER(_Q4),
                                        ctypes.POINTER(_Q4), _P, _I64, _P, _P, _P, _I]
        L.oracle_gdn_scan.argtypes = [_P, _P, _P, _P, _P, _P, _I64, _I, _I, _I, _P, _P, _I]
        for fn in ("oracle_gdn_scan", "oracle_router_logits_f64", "oracle_router_logits_f32", "oracle_select",
                   "oracle_route_structure", "oracle_expert_ffn", "oracle_forward",
                   "oracle_dequant_q4", "oracle_forward_q4"):
            getattr(L, fn).restype = _I
        _lib = L
    return _lib


def _threads(n):
    if n is not None:
        return int(n)
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return os.cpu_count() or 1


def _u16(a):
    return np.ascontiguousarray(a, dtype=np.uint16)


def _ptr(a):
    return None if a is None else a.ctypes.data


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"{what} failed with status {rc}")


def router_logits_f64(x, w_r, bias=None, nthreads=None):
    x, w_r = _u16(x), _u16(w_r)
    T, d = x.shape
    E = w_r.shape[0]
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    out = np.empty((T, E), dtype=np.float64)
    _check(lib().oracle_router_logits_f64(_ptr(x), T, d, _ptr(w_r), E, _ptr(b), _ptr(out),
                                          _threads(nthreads)), "router_logits_f64")
    return out


def router_logits_f32(x, w_r, bias=None, nthreads=None):
    x, w_r = _u16(x), _u16(w_r)
    T, d = x.shape
    E = w_r.shape[0]
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    out = np.empty((T, E), dtype=np.float32)
    _check(lib().oracle_router_logits_f32(_ptr(x), T, d, _ptr(w_r), E, _ptr(b), _ptr(out),
                                          _threads(nthreads)), "router_logits_f32")
    return out


def select(logits, k):
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    T, E = logits.shape
    idx = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float32)
    _check(lib().oracle_select(_ptr(logits), T, E, k, _ptr(idx), _ptr(w)), "select")
    return idx, w


def route_structure(topk_idx, E):
    topk_idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    T, k = topk_idx.shape
    counts = np.empty(E, dtype=np.int32)
    offsets = np.empty(E + 1, dtype=np.int32)
    perm = np.empty(T * k, dtype=np.int32)
    inv_perm = np.empty(T * k, dtype=np.int32)
    _check(lib().oracle_route_structure(_ptr(topk_idx), T, E, k, _ptr(counts), _ptr(offsets),
                                        _ptr(perm), _ptr(inv_perm)), "route_structure")
    return counts, offsets, perm, inv_perm


def route(x, w_r, k, bias=None, nthreads=None):
    """Routing of every token: dict with topk_idx, topk_w, counts, offsets, perm, inv_perm."""
    idx, w = select(router_logits_f32(x, w_r, bias, nthreads), k)
    counts, offsets, perm, inv_perm = route_structure(idx, w_r.shape[0])
    return dict(topk_idx=idx, topk_w=w, counts=counts, offsets=offsets, perm=perm,
                inv_perm=inv_perm)


def expert_ffn(x_row, w_gate, w_up, w_down):
    x_row, w_gate, w_up, w_down = map(_u16, (x_row, w_gate, w_up, w_down))
    f, d = w_gate.shape
    h = np.empty(f, dtype=np.float32)
    o = np.empty(d, dtype=np.float32)
    _check(lib().oracle_expert_ffn(_ptr(x_row), d, _ptr(w_gate), _ptr(w_up), _ptr(w_down), f,
                                   _ptr(h), _ptr(o)), "expert_ffn")
    return h, o


def forward(x, w_r, bias, experts, shared, k, tokens=None, nthreads=None):
    """Layer output rows (bf16 bits) for `tokens` (None: all tokens).

    experts: either a tuple of three arrays (w_gate [E][f][d], w_up [E][f][d],
    w_down [E][d][f]) or a dict {e: (w_gate_e, w_up_e, w_down_e)} holding at least every
    expert the listed tokens select.  shared: (ws_gate [fs][d], ws_up [fs][d], ws_down [d][fs]).
    Returns (y [n][d] uint16, topk_idx [n][k], topk_w [n][k]).
    """
    x, w_r = _u16(x), _u16(w_r)
    T, d = x.shape
    E = w_r.shape[0]
    keep = []
    ptrs = [(_P * E)(), (_P * E)(), (_P * E)()]
    if isinstance(experts, dict):
        items = experts.items()
        f = next(iter(experts.values()))[0].shape[0] if experts else 1
    else:
        items = ((e, (experts[0][e], experts[1][e], experts[2][e])) for e in range(E))
        f = experts[0].shape[1]
    for e, mats in items:
        for q in range(3):
            a = _u16(mats[q])
            keep.append(a)
            ptrs[q][int(e)] = a.ctypes.data
    sg, su, sd = map(_u16, shared)
    fs = sg.shape[0]
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    if tokens is None:
        tok = None
        n = T
    else:
        tok = np.ascontiguousarray(tokens, dtype=np.int64)
        n = tok.shape[0]
    y = np.empty((n, d), dtype=np.uint16)
    idx = np.empty((n, k), dtype=np.int32)
    w = np.empty((n, k), dtype=np.float32)
    dims = _Dims(d, E, k, f, fs)
    rc = lib().oracle_forward(ctypes.byref(dims), _ptr(x), T, _ptr(w_r), _ptr(b), ptrs[0], ptrs[1],
                              ptrs[2], _ptr(sg), _ptr(su), _ptr(sd), _ptr(tok), n, _ptr(y),
                              _ptr(idx), _ptr(w), _threads(nthreads))
    _check(rc, "forward")
    return y, idx, w


def _q4(m, keep):
    """(codes, scales, biases) arrays -> the C struct (arrays kept alive in `keep`)."""
    c = np.ascontiguousarray(m[0], dtype=np.uint8)
    sc, b = _u16(m[1]), _u16(m[2])
    keep += [c, sc, b]
    return _Q4(c.ctypes.data, sc.ctypes.data, b.ctypes.data)


def dequant_q4(codes, scales, biases):
    """fp32 weights [rows][K] of a 4-bit group-affine matrix (codes [rows][K/2] uint8,
    scales/biases [rows][K/64] bf16 bits)."""
    keep = []
    m = _q4((codes, scales, biases), keep)
    rows, K = int(np.prod(codes.shape[:-1])), codes.shape[-1] * 2
    out = np.empty((rows, K), dtype=np.float32)
    _check(lib().oracle_dequant_q4(ctypes.byref(m), rows, K, _ptr(out)), "dequant_q4")
    return out.reshape(codes.shape[:-1] + (K,))


def forward_q4(x, w_r, bias, experts, shared, k, tokens=None, nthreads=None):
    """forward() with 4-bit experts.  experts: {e: (gate, up, down)} holding at least every
    expert the listed tokens select, each matrix a (codes, scales, biases) triple; shared: the
    shared expert's three triples.  Returns (y [n][d] uint16, topk_idx, topk_w)."""
    x, w_r = _u16(x), _u16(w_r)
    T, d = x.shape
    E = w_r.shape[0]
    keep = []
    arrs = [(_Q4 * E)(), (_Q4 * E)(), (_Q4 * E)()]
    f = None
    for e, mats in experts.items():
        for q in range(3):
            arrs[q][int(e)] = _q4(mats[q], keep)
        f = np.asarray(mats[0][0]).shape[-2]
    sg, su, sd = (_q4(m, keep) for m in shared)
    fs = np.asarray(shared[0][0]).shape[-2]
    if f is None:
        f = fs
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    if tokens is None:
        tok, n = None, T
    else:
        tok = np.ascontiguousarray(tokens, dtype=np.int64)
        n = tok.shape[0]
    y = np.empty((n, d), dtype=np.uint16)
    idx = np.empty((n, k), dtype=np.int32)
    w = np.empty((n, k), dtype=np.float32)
    dims = _Dims(d, E, k, f, fs)
    rc = lib().oracle_forward_q4(ctypes.byref(dims), _ptr(x), T, _ptr(w_r), _ptr(b), arrs[0],
                                 arrs[1], arrs[2], ctypes.byref(sg), ctypes.byref(su),
                                 ctypes.byref(sd), _ptr(tok), n, _ptr(y), _ptr(idx), _ptr(w),
                                 _threads(nthreads))
    _check(rc, "forward_q4")
    return y, idx, w


def kth_gap(logits64, k):
    """Gap between the k-th and (k+1)-th largest logit of each row (fp64)."""
    part = -np.sort(-logits64, axis=1)
    return part[:, k - 1] - part[:, k]


def draw_x_with_gap(seed, layer, T, d, routers, k, min_gap=1e-3, max_rounds=64):
    """x [T][d] drawn by the seeded generator, every row redrawn (next redraw round of the
    same stream) until, for every (w_r, bias) in `routers`, the gap between its k-th and
    (k+1)-th largest fp64 logit is >= min_gap.  Returns (x, rounds, n_redraws)."""
    import synth
    rounds = np.zeros(T, dtype=np.int64)
    x = synth.x_rows(seed, layer, T, d, rounds)
    todo = np.arange(T)
    redraws = 0
    for _ in range(max_rounds):
        bad = np.zeros(todo.shape[0], dtype=bool)
        for w_r, bias in routers:
            bad |= kth_gap(router_logits_f64(x[todo], w_r, bias), k) < min_gap
        todo = todo[bad]
        if todo.size == 0:
            return x, rounds, redraws
        redraws += int(todo.size)
        rounds[todo] += 1
        for t in todo:
            x[t] = synth.normal_bf16(seed, synth.stream_id(synth.X, layer, int(rounds[t])),
                                     int(t) * d, d, synth.SIGMA_X)
    raise RuntimeError("gap rule not met after max_rounds redraws")


def gdn_scan(q, k, v, alpha, beta, s0=None, nthreads=None):
    """Gated DeltaNet scan (gdn_oracle.h): q, k [T][H][dk] and v [T][H][dv] bf16 bits, alpha,
    beta [T][H] fp32, s0 [H][dk][dv] fp32 or None (zeros).  Returns (o [T][H][dv], s [H][dk][dv])
    in fp64."""
    q, k, v = _u16(q), _u16(k), _u16(v)
    T, H, dk = q.shape
    dv = v.shape[2]
    assert k.shape == (T, H, dk) and v.shape == (T, H, dv)
    alpha = np.ascontiguousarray(alpha, dtype=np.float32)
    beta = np.ascontiguousarray(beta, dtype=np.float32)
    assert alpha.shape == (T, H) and beta.shape == (T, H)
    if s0 is not None:
        s0 = np.ascontiguousarray(s0, dtype=np.float32)
        assert s0.shape == (H, dk, dv)
    o = np.empty((T, H, dv), dtype=np.float64)
    s = np.empty((H, dk, dv), dtype=np.float64)
    _check(lib().oracle_gdn_scan(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta),
                                 None if s0 is None else _ptr(s0), T, H, dk, dv, _ptr(o),
                                 _ptr(s), _threads(nthreads)), "oracle_gdn_scan")
    return o, s
