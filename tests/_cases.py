"""Seeded test cases of the MoE layer: host inputs (for the oracle), device copies (for the
CUDA path), and oracle references.  Shapes follow the workloads of "Optimizing on-device
inference for Apple Silicon" (256 experts, top 8 plus one shared expert, prompts of 256 to
128K tokens, batch-1 decode); values come from the seeded generator in synth/.

x rows are drawn under the gap rule (oracle.draw_x_with_gap): the k-th and (k+1)-th router
logits of every token differ by at least 1e-3 in fp64, so both sides must select the same
experts even though their fp32 sums are ordered differently.
"""
from dataclasses import dataclass, field

import numpy as np

import oracle
import synth

TOL_REL = 2e-2   # max|gpu - ref| <= TOL_REL * max|ref| + TOL_ABS
TOL_ABS = 1e-3


@dataclass
class Case:
    name: str
    dims: synth.Dims
    T: int
    seed: int = 0
    layer: int = 0
    skew: bool = False
    x: np.ndarray = None          # [T][d] bf16 bits
    w_r: np.ndarray = None        # [E][d]
    bias: np.ndarray = None       # [E] fp32 or None
    host_w: dict = field(default_factory=dict)   # name -> full host array (when generated)
    redraws: int = 0


def build_case(name, d, f, fs, T, seed=0, layer=0, skew=False, full_host=True,
               w_r=None, bias=None):
    dims = synth.Dims(d=d, f=f, fs=fs)
    c = Case(name, dims, T, seed, layer, skew)
    c.w_r = synth.host_weight(seed, layer, "w_r", dims) if w_r is None else w_r
    if bias is not None:
        c.bias = bias
    elif skew:
        c.bias = synth.skew_bias(seed, layer, dims.E)
    if T > 0:
        c.x, _, c.redraws = oracle.draw_x_with_gap(seed, layer, T, d, [(c.w_r, c.bias)], dims.k)
    else:
        c.x = np.zeros((0, d), dtype=np.uint16)
    if full_host:
        for nm in synth.WEIGHT_NAMES:
            if nm != "w_r":
                c.host_w[nm] = synth.host_weight(seed, layer, nm, dims)
    return c


def expert_weights(c, experts):
    """{e: (w_gate_e, w_up_e, w_down_e)} for the listed experts (generated on demand)."""
    out = {}
    for e in experts:
        e = int(e)
        if c.host_w:
            out[e] = (c.host_w["w_gate"][e], c.host_w["w_up"][e], c.host_w["w_down"][e])
        else:
            out[e] = tuple(synth.host_weight(c.seed, c.layer, nm, c.dims, expert=e)
                           for nm in ("w_gate", "w_up", "w_down"))
    return out


def shared_weights(c):
    if c.host_w:
        return c.host_w["ws_gate"], c.host_w["ws_up"], c.host_w["ws_down"]
    return tuple(synth.host_weight(c.seed, c.layer, nm, c.dims)
                 for nm in ("ws_gate", "ws_up", "ws_down"))


def oracle_route(c):
    return oracle.route(c.x, c.w_r, c.dims.k, c.bias)


def oracle_outputs(c, tokens=None):
    """Oracle y rows (bf16 bits) for `tokens` (None: all)."""
    toks = np.arange(c.T) if tokens is None else np.asarray(tokens)
    idx, _ = oracle.select(oracle.router_logits_f32(c.x[toks], c.w_r, c.bias), c.dims.k)
    experts = expert_weights(c, np.unique(idx))
    y, _, _ = oracle.forward(c.x, c.w_r, c.bias, experts, shared_weights(c), c.dims.k,
                             tokens=toks)
    return y


def sample_tokens(T, n_edge=64, stride=17):
    """First and last n_edge tokens plus every stride-th token."""
    s = set(range(min(T, n_edge))) | set(range(max(0, T - n_edge), T)) | set(range(0, T, stride))
    return np.array(sorted(s), dtype=np.int64)


# ---------------------------------------------------------------- device side

def to_device(c):
    """Device tensors of the case's weights (generated on the device by the same generator
    when the host copy is absent) and of x."""
    import torch
    dev = torch.device("cuda")
    W = {}
    for nm in synth.WEIGHT_NAMES:
        shape = synth.weight_shape(nm, c.dims)
        if nm == "w_r":
            W[nm] = torch.from_numpy(c.w_r.view(np.int16)).to(dev).view(torch.bfloat16)
        elif nm in c.host_w:
            W[nm] = torch.from_numpy(c.host_w[nm].view(np.int16)).to(dev).view(torch.bfloat16)
        else:
            t = torch.empty(shape, dtype=torch.bfloat16, device=dev)
            synth.device_weight(c.seed, c.layer, nm, c.dims, t.data_ptr(),
                                torch.cuda.current_stream().cuda_stream)
            W[nm] = t
    W["w_router"] = W.pop("w_r")
    if c.bias is not None:
        W["router_bias"] = torch.from_numpy(c.bias).to(dev)
    x = torch.from_numpy(c.x.view(np.int16)).to(dev).view(torch.bfloat16)
    return W, x


def bf16_bits(t):
    """uint16 numpy view of a bf16 torch tensor."""
    return t.detach().cpu().view(__import__("torch").int16).numpy().view(np.uint16)


def assert_close(y_gpu_bits, y_ref_bits, what=""):
    g = synth.bf16_to_f32(y_gpu_bits).astype(np.float64)
    r = synth.bf16_to_f32(y_ref_bits).astype(np.float64)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU output"
    err = np.max(np.abs(g - r)) if g.size else 0.0
    bound = TOL_REL * (np.max(np.abs(r)) if r.size else 0.0) + TOL_ABS
    assert err <= bound, f"{what}: max|gpu-ref| = {err:.3e} > {bound:.3e}"
    return err, bound


# ---------------------------------------------------------------- 4-bit experts

def q4_to_device(c):
    """Device tensors of the case's 4-bit experts (generated on the device) and bf16 router."""
    import torch
    dev = torch.device("cuda")
    W = {"w_router": torch.from_numpy(c.w_r.view(np.int16)).to(dev).view(torch.bfloat16)}
    s = torch.cuda.current_stream().cuda_stream
    for nm in synth.Q4_NAMES:
        cs, gs = synth.q4_shapes(nm, c.dims)
        codes = torch.empty(cs, dtype=torch.uint8, device=dev)
        sc = torch.empty(gs, dtype=torch.bfloat16, device=dev)
        b = torch.empty(gs, dtype=torch.bfloat16, device=dev)
        synth.q4_device(c.seed, c.layer, nm, c.dims, codes.data_ptr(), sc.data_ptr(),
                        b.data_ptr(), s)
        W[nm] = (codes, sc, b)
    if c.bias is not None:
        W["router_bias"] = torch.from_numpy(c.bias).to(dev)
    return W


def oracle_outputs_q4(c, tokens=None):
    """Oracle y rows (bf16 bits) of the case with 4-bit experts (only the selected experts'
    weights are generated on the host)."""
    toks = np.arange(c.T) if tokens is None else np.asarray(tokens)
    idx, _ = oracle.select(oracle.router_logits_f32(c.x[toks], c.w_r, c.bias), c.dims.k)
    experts = {int(e): tuple(synth.q4_host(c.seed, c.layer, nm, c.dims, expert=int(e))
                             for nm in ("w_gate", "w_up", "w_down")) for e in np.unique(idx)}
    shared = tuple(synth.q4_host(c.seed, c.layer, nm, c.dims)
                   for nm in ("ws_gate", "ws_up", "ws_down"))
    y, _, _ = oracle.forward_q4(c.x, c.w_r, c.bias, experts, shared, c.dims.k, tokens=toks)
    return y
