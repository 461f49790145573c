"""Argument checks of the Python binding, on the CPU.

The C ABI takes plain pointers and one (rows, cols) pair per matrix, so it
reads G[i] and reads and writes M[i] over rows x cols elements whatever their
allocation holds: the binding must refuse a G or M that does not have W's
shape before anything reaches the library.  Shapes are checked before device
placement, so these cases run on CPU tensors; a well-formed call on CPU
tensors must then stop at the device check (the product never computes on the
host).
"""
import pytest
import torch

import muon_newton_schulz_step_gb300 as mg
from muon_newton_schulz_step_gb300 import optim


def _wgm(shape=(8, 16), g_shape=None, m_shape=None):
    W = torch.zeros(shape, dtype=torch.bfloat16)
    G = torch.zeros(g_shape or shape, dtype=torch.bfloat16)
    M = torch.zeros(m_shape or shape, dtype=torch.float32)
    return [W], [G], [M]


STEP_CALLS = {
    "muon_step": lambda W, G, M: mg.muon_step(W, G, M, 0.02, 0.95, 0.1),
    "muon_step_ex": lambda W, G, M: mg.muon_step_ex(W, G, M, 0.02, 0.95, 0.1),
    "MuonStepBatch": lambda W, G, M: mg.MuonStepBatch(W, G, M),
    "MuonHostStep": lambda W, G, M: mg.MuonHostStep(W, G, M),
}


@pytest.mark.parametrize("call", list(STEP_CALLS))
@pytest.mark.parametrize("bad", [
    dict(m_shape=(8, 8)),            # M smaller than W
    dict(m_shape=(16, 8)),           # M transposed
    dict(g_shape=(8, 8)),            # G smaller than W
    dict(g_shape=(16, 8)),           # G transposed
    dict(g_shape=(2, 16, 8)),        # stacked G with the wrong trailing shape
])
def test_mismatched_g_or_m_is_refused(call, bad):
    W, G, M = _wgm(**bad)
    with pytest.raises(ValueError, match=r"[GM]\[0\] has shape"):
        STEP_CALLS[call](W, G, M)


@pytest.mark.parametrize("call", list(STEP_CALLS))
def test_length_and_rank_checks(call):
    W, G, M = _wgm()
    with pytest.raises(ValueError, match="same length"):
        STEP_CALLS[call](W + W, G, M)
    with pytest.raises(ValueError, match=r"W\[0\] must be 2-D"):
        STEP_CALLS[call]([W[0].unsqueeze(0)], [G[0].unsqueeze(0)], [M[0].unsqueeze(0)])
    with pytest.raises(ValueError, match="must be a tensor"):
        STEP_CALLS[call]([W[0]], [None], [M[0]])


def test_stacked_gradients_only_where_the_call_takes_them():
    W, G, M = _wgm(g_shape=(3, 8, 16))
    with pytest.raises(ValueError, match=r"G\[0\] has shape"):
        mg.muon_step(W, G, M, 0.02, 0.95, 0.1)
    with pytest.raises(ValueError, match="CUDA tensor"):        # shapes pass, device does not
        mg.muon_step_ex(W, G, M, 0.02, 0.95, 0.1)


@pytest.mark.parametrize("call", ["muon_step", "muon_step_ex", "MuonStepBatch"])
def test_host_tensors_stop_at_the_device_check(call):
    with pytest.raises(ValueError, match="CUDA tensor"):
        STEP_CALLS[call](*_wgm())


def test_host_step_wants_pinned_memory():
    with pytest.raises(ValueError, match="pinned"):
        mg.MuonHostStep(*_wgm())


def test_ns_and_adamw_refuse_host_tensors():
    x = torch.zeros(8, 16, dtype=torch.bfloat16)
    for fn in (mg.muon_ns5_batched, mg.muon_ns_batched_ex, mg.muon_ns5_batched_static):
        with pytest.raises(ValueError, match="CUDA tensor"):
            fn([x])
    p = torch.zeros(16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        mg.muon_adamw_step([p], [p.clone()], [p.clone()], [p.clone()], lr=1e-3, step=1)
    with pytest.raises(ValueError, match="same length"):
        mg.muon_adamw_step([p], [], [p.clone()], [p.clone()], lr=1e-3, step=1)


def test_coefficient_schedule_shape():
    assert mg._schedule(None, 5) == (None, 0)
    arr, per_step = mg._schedule((1.0, 2.0, 3.0), 5)
    assert per_step == 0 and list(arr) == [1.0, 2.0, 3.0]
    arr, per_step = mg._schedule([(1, 2, 3), (4, 5, 6)], 2)
    assert per_step == 1 and list(arr) == [1, 2, 3, 4, 5, 6]
    with pytest.raises(ValueError, match="one \\(a, b, c\\) triple per step"):
        mg._schedule([(1, 2, 3), (4, 5, 6)], 3)
    with pytest.raises(ValueError, match="one \\(a, b, c\\) triple per step"):
        mg._schedule([(1, 2, 3), (4, 5)], 2)
    with pytest.raises(ValueError, match="coeffs must be"):
        mg._schedule((1.0, 2.0), 5)


def test_optimizer_routes_matrices_to_muon_and_checks_rank():
    mat = torch.nn.Parameter(torch.zeros(8, 16))
    vec = torch.nn.Parameter(torch.zeros(16))
    opt = optim.MuonAdamW([{"params": [mat, vec]}])
    group = opt.param_groups[0]
    assert opt._is_muon(group, mat) and not opt._is_muon(group, vec)
    forced = optim.MuonAdamW([{"params": [vec], "use_muon": True}])
    vec.grad = torch.zeros(16)
    with pytest.raises(ValueError, match="matrices"):
        forced.step()
    mat.grad = torch.zeros(8, 16)
    with pytest.raises(ValueError, match="CUDA tensor"):    # no host computation
        opt.step()
