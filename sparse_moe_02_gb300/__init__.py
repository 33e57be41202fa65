"""Python binding of libmoe, the GB300 (sm_103a) mixture-of-experts FFN layer.

Argument marshalling only: every function here forwards to the C entry point of the same
name declared in include/moe.h and returns its status code; all arithmetic runs in the CUDA
kernels of libmoe.so.  There is no fallback: if the library is missing or cannot be loaded,
import-time use fails loudly.

MoeLayer is a small convenience wrapper that takes torch CUDA tensors (PyTorch is used only
for device memory and streams) and raises MoeError on a non-zero status.

With MOE_DEBUG_LIBRARY=1 in the environment the binding loads libmoe_debug.so instead: the same
library built with MOE_DEBUG, which checks every routing it produces (moe_check_routing) and
records a failure in the handle's device error word.
"""
import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_debug.so" if os.environ.get("MOE_DEBUG_LIBRARY") == "1"
                        else "libmoe.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_ALIGNMENT = 3
MOE_ERR_CUDA = 4
MOE_ERR_TIMEOUT = 5
MOE_ERR_DEVICE = 6
MOE_ERR_NO_MEMORY = 7

MOE_SCHEDULE_AUTO = 0
MOE_SCHEDULE_GEMM = 1
MOE_SCHEDULE_GEMV = 2

EXPORTS = ("moe_create", "moe_route", "moe_forward", "moe_forward_host", "moe_get_device_error",
           "moe_destroy", "moe_status_string", "moe_last_cuda_error", "moe_profile_begin",
           "moe_profile_end", "moe_route_one_noalloc", "moe_create_q4", "moe_read_probe",
           "moe_test_expire_waits", "gdn_scan", "moe_check_routing")

# kernel order reported by moe_profile_end
KERNELS_GEMM = ("router_topk", "route_plan_scatter", "experts", "combine")
KERNELS_GEMV = ("decode_router_shared", "decode_gateup", "decode_down_combine")

_c_int, _c_void_p = ctypes.c_int, ctypes.c_void_p


class moe_config(ctypes.Structure):
    _fields_ = [("d", _c_int), ("n_experts", _c_int), ("top_k", _c_int), ("ffn_dim", _c_int),
                ("shared_ffn_dim", _c_int), ("max_tokens", _c_int), ("schedule", _c_int),
                ("chunk_tokens", _c_int)]


class moe_weights(ctypes.Structure):
    _fields_ = [("w_router", _c_void_p), ("router_bias", _c_void_p), ("w_gate", _c_void_p),
                ("w_up", _c_void_p), ("w_down", _c_void_p), ("ws_gate", _c_void_p),
                ("ws_up", _c_void_p), ("ws_down", _c_void_p)]


class moe_q4_matrix(ctypes.Structure):
    _fields_ = [("codes", _c_void_p), ("scales", _c_void_p), ("biases", _c_void_p)]


class moe_weights_q4(ctypes.Structure):
    _fields_ = [("w_router", _c_void_p), ("router_bias", _c_void_p),
                ("w_gate", moe_q4_matrix), ("w_up", moe_q4_matrix), ("w_down", moe_q4_matrix),
                ("ws_gate", moe_q4_matrix), ("ws_up", moe_q4_matrix),
                ("ws_down", moe_q4_matrix)]


_lib = None


def lib():
    """The loaded libmoe.so (raises OSError if it is not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise OSError(f"{os.path.basename(LIB_PATH)} not built ({LIB_PATH}); "
                          "run __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        L.moe_create.argtypes = [ctypes.POINTER(moe_config), ctypes.POINTER(moe_weights),
                                 ctypes.POINTER(_c_void_p)]
        L.moe_read_probe.argtypes = [_c_void_p, ctypes.c_size_t, _c_void_p, _c_void_p]
        L.moe_create_q4.argtypes = [ctypes.POINTER(moe_config), ctypes.POINTER(moe_weights_q4),
                                    ctypes.POINTER(_c_void_p)]
        L.moe_route.argtypes = [_c_void_p, _c_void_p, _c_int, _c_void_p, _c_void_p, _c_void_p,
                                _c_void_p, _c_void_p]
        L.moe_forward.argtypes = [_c_void_p, _c_void_p, _c_int, _c_void_p, _c_void_p]
        L.moe_forward_host.argtypes = [_c_void_p, _c_void_p, _c_int, _c_void_p, _c_void_p]
        L.moe_get_device_error.argtypes = [_c_void_p, _c_void_p]
        L.moe_destroy.argtypes = [_c_void_p]
        L.moe_status_string.argtypes = [_c_int]
        L.moe_status_string.restype = ctypes.c_char_p
        L.moe_last_cuda_error.argtypes = []
        L.moe_profile_begin.argtypes = [_c_void_p, _c_int]
        L.moe_profile_end.argtypes = [_c_void_p, ctypes.POINTER(ctypes.c_float), _c_int,
                                      ctypes.POINTER(_c_int), ctypes.POINTER(_c_int)]
        L.moe_route_one_noalloc.argtypes = [_c_void_p, _c_int, _c_void_p, _c_void_p, _c_void_p,
                                            _c_void_p, _c_void_p]
        L.moe_test_expire_waits.argtypes = [_c_void_p, _c_int]
        L.moe_check_routing.argtypes = [_c_void_p, _c_void_p, _c_void_p, _c_int, _c_void_p,
                                        _c_void_p]
        L.gdn_scan.argtypes = [_c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p,
                               _c_void_p, _c_void_p, ctypes.c_int64, _c_int, _c_int, _c_int,
                               _c_void_p]
        for fn in ("moe_create", "moe_create_q4", "moe_read_probe", "moe_route", "moe_forward", "moe_forward_host",
                   "moe_get_device_error", "moe_destroy", "moe_last_cuda_error",
                   "moe_profile_begin", "moe_profile_end", "moe_route_one_noalloc",
                   "moe_test_expire_waits", "gdn_scan", "moe_check_routing"):
            getattr(L, fn).restype = _c_int
        _lib = L
    return _lib


def moe_create(cfg, weights):
    """Returns (status, handle)."""
    h = _c_void_p()
    st = lib().moe_create(ctypes.byref(cfg), ctypes.byref(weights), ctypes.byref(h))
    return st, h


def moe_create_q4(cfg, weights_q4):
    """Returns (status, handle) for 4-bit experts (moe_weights_q4)."""
    h = _c_void_p()
    st = lib().moe_create_q4(ctypes.byref(cfg), ctypes.byref(weights_q4), ctypes.byref(h))
    return st, h


def moe_read_probe(buf, nbytes, sink, stream):
    return lib().moe_read_probe(buf, nbytes, sink, stream)


def moe_route(h, x, T, topk_idx, topk_w, offsets, perm, stream):
    return lib().moe_route(h, x, T, topk_idx, topk_w, offsets, perm, stream)


def moe_forward(h, x, T, y, stream):
    return lib().moe_forward(h, x, T, y, stream)


def moe_forward_host(h, x_host, T, y_host, stream):
    return lib().moe_forward_host(h, x_host, T, y_host, stream)


def moe_get_device_error(h, stream):
    return lib().moe_get_device_error(h, stream)


def moe_destroy(h):
    return lib().moe_destroy(h)


def moe_status_string(status):
    return lib().moe_status_string(status).decode()


def moe_last_cuda_error():
    return lib().moe_last_cuda_error()


def moe_route_one_noalloc(x, d, w_router, router_bias, topk_idx, topk_w, stream):
    """Routing of one token with no device allocation (see include/moe.h)."""
    return lib().moe_route_one_noalloc(x, d, w_router, router_bias, topk_idx, topk_w, stream)


def moe_check_routing(topk_idx, offsets, perm, T, status, stream):
    """Consistency check of a routing (see include/moe.h); *status (a device int) ends as
    MOE_OK or MOE_ERR_DEVICE once the stream has run."""
    return lib().moe_check_routing(topk_idx, offsets, perm, T, status, stream)


def gdn_scan(q, k, v, alpha, beta, state_in, state_out, o, T, H, dk, dv, stream):
    """Gated DeltaNet recurrent scan over T tokens of H heads (see include/gdn.h); device
    pointers, state_in may be None (zero state)."""
    return lib().gdn_scan(q, k, v, alpha, beta, state_in, state_out, o, T, H, dk, dv, stream)


def moe_test_expire_waits(h, n_calls):
    """Test hook: the next n_calls batch-1 forwards time out at their grid barrier (see
    include/moe.h)."""
    return lib().moe_test_expire_waits(h, n_calls)


def moe_profile_begin(h, n_calls):
    return lib().moe_profile_begin(h, n_calls)


def moe_profile_end(h):
    """Returns (status, [ms per kernel summed over the recorded calls], n_calls)."""
    ms = (ctypes.c_float * 8)()
    nk, nc = _c_int(), _c_int()
    st = lib().moe_profile_end(h, ms, 8, ctypes.byref(nk), ctypes.byref(nc))
    return st, list(ms)[:nk.value], nc.value


class MoeError(RuntimeError):
    def __init__(self, status, what):
        detail = moe_status_string(status)
        if status == MOE_ERR_CUDA:
            detail += f" (cudaError {moe_last_cuda_error()})"
        super().__init__(f"{what}: {detail}")
        self.status = status


def _check(status, what):
    if status != MOE_OK:
        raise MoeError(status, what)


def _ptr(t):
    return None if t is None else t.data_ptr()


class MoeLayer:
    """One MoE layer over torch CUDA tensors (bf16 weights, layouts as in include/moe.h).

    weights: dict with w_router [E][d], w_gate/w_up [E][f][d], w_down [E][d][f],
    ws_gate/ws_up [fs][d], ws_down [d][fs] (bf16, contiguous, on the current device) and
    optionally router_bias [E] (float32).  The tensors are borrowed: keep them alive.
    """

    def __init__(self, weights, max_tokens, schedule=MOE_SCHEDULE_AUTO, chunk_tokens=0):
        if isinstance(weights["w_gate"], tuple):
            self._init_q4(weights, max_tokens, schedule, chunk_tokens)
            return
        E, f, d = weights["w_gate"].shape
        fs = weights["ws_gate"].shape[0]
        self.d, self.f, self.fs, self.E, self.k = d, f, fs, E, 8
        self.max_tokens = max_tokens
        self._weights = weights  # keep the borrowed tensors alive
        cfg = moe_config(d, E, 8, f, fs, max_tokens, schedule, chunk_tokens)
        w = moe_weights(_ptr(weights["w_router"]), _ptr(weights.get("router_bias")),
                        _ptr(weights["w_gate"]), _ptr(weights["w_up"]), _ptr(weights["w_down"]),
                        _ptr(weights["ws_gate"]), _ptr(weights["ws_up"]),
                        _ptr(weights["ws_down"]))
        st, self.handle = moe_create(cfg, w)
        _check(st, "moe_create")

    def _init_q4(self, weights, max_tokens, schedule, chunk_tokens):
        """4-bit experts: each expert tensor is a (codes uint8, scales bf16, biases bf16)
        triple of torch tensors, shapes as in synth.q4_shapes; w_router stays bf16."""
        codes = weights["w_gate"][0]
        E, f, d = codes.shape[0], codes.shape[1], codes.shape[2] * 2
        fs = weights["ws_gate"][0].shape[0]
        self.d, self.f, self.fs, self.E, self.k = d, f, fs, E, 8
        self.max_tokens = max_tokens
        self._weights = weights

        def m(name):
            c, sc, b = weights[name]
            return moe_q4_matrix(_ptr(c), _ptr(sc), _ptr(b))

        cfg = moe_config(d, E, 8, f, fs, max_tokens, schedule, chunk_tokens)
        w = moe_weights_q4(_ptr(weights["w_router"]), _ptr(weights.get("router_bias")),
                           m("w_gate"), m("w_up"), m("w_down"), m("ws_gate"), m("ws_up"),
                           m("ws_down"))
        st, self.handle = moe_create_q4(cfg, w)
        _check(st, "moe_create_q4")

    @staticmethod
    def _stream(stream):
        import torch
        s = torch.cuda.current_stream() if stream is None else stream
        return s.cuda_stream

    def forward(self, x, y=None, stream=None):
        import torch
        T = x.shape[0]
        if y is None:
            y = torch.empty_like(x)
        _check(moe_forward(self.handle, _ptr(x), T, _ptr(y), self._stream(stream)), "moe_forward")
        return y

    def forward_host(self, x_host, y_host, stream=None):
        _check(moe_forward_host(self.handle, _ptr(x_host), x_host.shape[0], _ptr(y_host),
                                self._stream(stream)), "moe_forward_host")
        return y_host

    def route(self, x, stream=None):
        import torch
        T = x.shape[0]
        dev = x.device
        out = dict(topk_idx=torch.empty((T, 8), dtype=torch.int32, device=dev),
                   topk_w=torch.empty((T, 8), dtype=torch.float32, device=dev),
                   offsets=torch.empty(self.E + 1, dtype=torch.int32, device=dev),
                   perm=torch.empty(T * 8, dtype=torch.int32, device=dev))
        _check(moe_route(self.handle, _ptr(x), T, _ptr(out["topk_idx"]), _ptr(out["topk_w"]),
                         _ptr(out["offsets"]), _ptr(out["perm"]), self._stream(stream)),
               "moe_route")
        return out

    def device_error(self, stream=None):
        return moe_get_device_error(self.handle, self._stream(stream))

    def close(self):
        if self.handle:
            _check(moe_destroy(self.handle), "moe_destroy")
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
