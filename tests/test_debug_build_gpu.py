"""The GDN_DEBUG build (libgdn_debug) on the GPU: the same results as the
release build bit for bit when the inputs meet the documented preconditions
(its device-side index checks never misfire on the fused, separate and
many-sequence paths), and GDN_ERR_INVALID_ARG from
gdn_chunk_prefill_device_status when they do not: g > 0 or not finite, beta
outside [0, 1], a q or k row not of unit norm.  The release build does not
check these (and still runs).  These checks stand in for the compute
sanitizer, which this GPU pool does not offer."""
import ctypes

import pytest
import torch

import gated_deltanet_linear_chunk_gb300 as gdn
from gated_deltanet_linear_chunk_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def libs():
    import __graft_entry__
    __graft_entry__.build()
    return gdn.library(), gdn.debug_library()


def run(lib, p):
    """One prefill through `lib`'s C ABI; returns (call status, device
    status, out, final state)."""
    dev = torch.device("cuda")
    T, Hk, dk = p.q.shape
    Hv, dv = p.v.shape[1:]
    N = p.cu_seqlens.shape[0] - 1
    prob = gdn.make_problem(N, T, Hk, Hv, dk, dv, torch.bfloat16)
    need = lib.gdn_chunk_prefill_workspace_size(ctypes.byref(prob))
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device=dev)
    prob = gdn.make_problem(N, T, Hk, Hv, dk, dv, torch.bfloat16, ws)
    args = [x.to(dev) for x in (p.q, p.k, p.v, p.g, p.beta, p.cu_seqlens)]
    h0 = None if p.initial_state is None else p.initial_state.to(dev)
    out = torch.full((T, Hv, dv), float("nan"), dtype=torch.bfloat16, device=dev)
    fin = torch.full((N, Hv, dv, dk), float("nan"), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    rc = lib.gdn_chunk_prefill(ctypes.byref(prob), *[a.data_ptr() for a in args],
                               None if h0 is None else h0.data_ptr(), out.data_ptr(),
                               fin.data_ptr(), stream)
    torch.cuda.synchronize()
    st = lib.gdn_chunk_prefill_device_status(ws.data_ptr(), stream)
    return rc, st, out, fin


@pytest.mark.parametrize("lens,Hk,Hv", [
    ([300, 1, 64, 0, 77, 200], 2, 6),     # separate kernels, ragged, empty sequence
    ([4000], 16, 48),                      # fused kernel
    ([700, 900], 4, 12),                   # fused kernel over two sequences
])
def test_debug_build_matches_release(libs, lens, Hk, Hv):
    rel, dbg = libs
    p = inputs.prefill_inputs(lens, Hk, Hv, 128, 128, dtype=torch.bfloat16, seed=61,
                              initial_state_std=0.02)
    r = run(rel, p)
    d = run(dbg, p)
    assert r[:2] == (gdn.GDN_OK, gdn.GDN_OK) and d[:2] == (gdn.GDN_OK, gdn.GDN_OK)
    assert torch.equal(r[2], d[2]), "output differs between the release and debug builds"
    assert torch.equal(r[3], d[3]), "final state differs between the release and debug builds"


def _g_positive(p): p.g[5, 2] = 0.1
def _g_nan(p): p.g[7, 0] = float("nan")
def _beta_above_one(p): p.beta[3, 1] = 1.5
def _beta_negative(p): p.beta[100, 4] = -0.25
def _q_not_unit(p): p.q[10, 0] = (p.q[10, 0].float() * 2).to(p.q.dtype)
def _k_not_unit(p): p.k[211, 1] = (p.k[211, 1].float() * 0.5).to(p.k.dtype)


@pytest.mark.parametrize("mutate", [_g_positive, _g_nan, _beta_above_one, _beta_negative,
                                    _q_not_unit, _k_not_unit])
def test_debug_build_reports_inputs_outside_the_preconditions(libs, mutate):
    rel, dbg = libs
    p = inputs.prefill_inputs([150, 90], 2, 6, 128, 128, dtype=torch.bfloat16, seed=62)
    mutate(p)
    rc, st, _, _ = run(dbg, p)
    assert rc == gdn.GDN_OK
    assert st == gdn.GDN_ERR_INVALID_ARG, gdn.gdn_status_string(st)
    rc, st, _, _ = run(rel, p)
    assert (rc, st) == (gdn.GDN_OK, gdn.GDN_OK)  # (the release build does not check)
