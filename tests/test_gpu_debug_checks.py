"""The routing consistency check (moe_check_routing) and the debug build that runs it inside
every routing (libmoe_debug.so, compiled with MOE_DEBUG).

- Routings the library produces pass: the tensor-core schedule at T = 300 (tiny shape) and
  T = 4096 (the benchmark shape), the matrix-vector router at T = 1 and T = 5.
- Each broken invariant, planted on the host into a copy of a valid routing, is reported as
  MOE_ERR_DEVICE: an expert id out of range, ids not ascending or repeated within a token,
  offsets not starting at 0, not ending at 8T or not monotone, a perm entry out of range, two
  perm entries swapped across groups or within a group, a perm entry repeated.  The arrays keep
  their exact sizes; the check reads nothing outside them whatever they hold.
- The debug library (in a child process) runs the same layers with its checks on and reports
  no device error, with outputs within the oracle bar.
"""
import os
import subprocess
import sys

import numpy as np
import pytest

import sparse_moe_02_gb300 as moe
from _cases import build_case, to_device

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("CUDA GPU required for -m gpu tests")
    yield
    torch.cuda.synchronize()


def _check(topk_idx, offsets, perm, T):
    """moe_check_routing on device copies of host int32 arrays; returns the status it wrote."""
    import torch
    ti = torch.from_numpy(np.ascontiguousarray(topk_idx, dtype=np.int32)).cuda()
    of = torch.from_numpy(np.ascontiguousarray(offsets, dtype=np.int32)).cuda()
    pm = torch.from_numpy(np.ascontiguousarray(perm, dtype=np.int32)).cuda()
    status = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    st = moe.moe_check_routing(ti.data_ptr(), of.data_ptr(), pm.data_ptr(), T, status.data_ptr(),
                               torch.cuda.current_stream().cuda_stream)
    assert st == moe.MOE_OK, moe.moe_status_string(st)
    return int(status.cpu()[0])


SHAPES = {"tiny": (512, 128, 128), "bench": (2048, 512, 512)}


def _route(case_name, T, schedule=moe.MOE_SCHEDULE_AUTO):
    d, f, fs = SHAPES[case_name]
    c = build_case(case_name, d, f, fs, T, seed=T, full_host=case_name == "tiny")
    W, x = to_device(c)
    L = moe.MoeLayer(W, T, schedule=schedule)
    r = L.route(x)
    import torch
    torch.cuda.synchronize()
    assert L.device_error() == moe.MOE_OK
    out = {k: v.cpu().numpy() for k, v in r.items()}
    L.close()
    return out


@pytest.mark.parametrize("case_name,T", [("tiny", 300), ("bench", 4096), ("bench", 1),
                                         ("tiny", 5)])
def test_library_routing_passes(case_name, T):
    r = _route(case_name, T)
    assert _check(r["topk_idx"].reshape(-1), r["offsets"], r["perm"], T) == moe.MOE_OK


def _planted(name, idx, off, perm):
    idx, off, perm = idx.copy(), off.copy(), perm.copy()
    n = idx.size
    if name == "id_too_large":
        idx[13] = 256
    elif name == "id_negative":
        idx[21] = -1
    elif name == "ids_not_ascending":
        idx[8], idx[9] = idx[9], idx[8]
    elif name == "id_repeated":
        idx[17] = idx[16]
    elif name == "offsets_not_from_zero":
        off[0] = 1
    elif name == "offsets_wrong_total":
        off[-1] = n - 1
    elif name == "offsets_not_monotone":
        e = int(np.flatnonzero(np.diff(off) > 0)[0])  # first non-empty group
        off[e + 1] = off[e + 2] + 1 if off[e + 2] + 1 < n else n - 1
        off[e + 2] = off[e + 1] - 2
    elif name == "perm_out_of_range":
        perm[5] = n
    elif name == "perm_negative":
        perm[6] = -3
    elif name == "perm_swapped_across_groups":
        a, b = int(off[1] - 1), int(off[1])  # last slot of one group, first of the next
        g = np.searchsorted(off, np.arange(n), side="right") - 1
        assert g[a] != g[b]
        perm[a], perm[b] = perm[b], perm[a]
    elif name == "perm_swapped_within_group":
        g = np.diff(off)
        e = int(np.flatnonzero(g >= 2)[0])
        a = int(off[e])
        perm[a], perm[a + 1] = perm[a + 1], perm[a]
    elif name == "perm_repeated":
        g = np.diff(off)
        e = int(np.flatnonzero(g >= 2)[0])
        a = int(off[e])
        perm[a + 1] = perm[a]
    else:
        raise ValueError(name)
    return idx, off, perm


PLANTED = ["id_too_large", "id_negative", "ids_not_ascending", "id_repeated",
           "offsets_not_from_zero", "offsets_wrong_total", "offsets_not_monotone",
           "perm_out_of_range", "perm_negative", "perm_swapped_across_groups",
           "perm_swapped_within_group", "perm_repeated"]


@pytest.fixture(scope="module")
def tiny_routing():
    r = _route("tiny", 64)
    return r["topk_idx"].reshape(-1).astype(np.int32), r["offsets"].astype(np.int32), \
        r["perm"].astype(np.int32)


@pytest.mark.parametrize("name", PLANTED)
def test_each_broken_invariant_is_reported(tiny_routing, name):
    idx, off, perm = tiny_routing
    assert _check(idx, off, perm, 64) == moe.MOE_OK
    assert _check(*_planted(name, idx, off, perm), 64) == moe.MOE_ERR_DEVICE


CHILD = r"""
import sys
import numpy as np
import torch
sys.path.insert(0, sys.argv[1])
sys.path.insert(0, sys.argv[1] + "/tests")
import sparse_moe_02_gb300 as moe
from _cases import build_case, oracle_outputs, to_device, assert_close, bf16_bits
assert moe.LIB_PATH.endswith("libmoe_debug.so"), moe.LIB_PATH
shapes = {"tiny": (512, 128, 128), "bench": (2048, 512, 512)}
for name, T, sched in (("tiny", 300, moe.MOE_SCHEDULE_AUTO), ("bench", 1, moe.MOE_SCHEDULE_AUTO),
                       ("tiny", 5, moe.MOE_SCHEDULE_GEMM), ("tiny", 1, moe.MOE_SCHEDULE_GEMM)):
    d, f, fs = shapes[name]
    c = build_case(name, d, f, fs, T, seed=T, full_host=name == "tiny")
    W, x = to_device(c)
    L = moe.MoeLayer(W, T, schedule=sched)
    y = L.forward(x)
    L.route(x)
    torch.cuda.synchronize()
    assert L.device_error() == moe.MOE_OK, (name, T)
    assert_close(bf16_bits(y), oracle_outputs(c))
    L.close()
print("debug library ok")
"""


def test_debug_library_checks_every_routing_and_stays_clean():
    env = dict(os.environ, MOE_DEBUG_LIBRARY="1")
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], env=env, capture_output=True,
                       text=True, timeout=900)
    assert r.returncode == 0 and "debug library ok" in r.stdout, r.stdout[-2000:] + r.stderr[-3000:]
