"""Bounded device-side waits run out, report BS_ERR_TIMEOUT and leave the GPU usable.

The fused decode step's attention waits for each unit's selection to be published by
the front kernel. Here one unit's selection ticket in the caller-owned workspace is set
so far past its count that no CTA of the front kernel ever elects itself to select that
unit: its selection is never published. With the wait limit shortened to 2 ms through
the public knob, the attention's wait gives up, the kernels finish, and the status word
reads BS_ERR_TIMEOUT. Nothing faults: the failure is made on the host, in a buffer the
caller owns. After zeroing the workspace, the same layer runs the step again and
matches the float64 oracle.

The layer here (8 units) takes the plan whose front kernel elects a selecting CTA per
unit through those tickets. The plan for more than 2048 candidates a unit selects every
unit in a kernel of its own (one CTA per unit, no tickets), so no buffer the caller owns
can hold a selection back there; its attention waits through the same bounded wait
function.
"""
import numpy as np
import pytest
import torch

from long_context_serving_gb300 import bsattn as B
from long_context_serving_gb300.build import build
from long_context_serving_gb300.layer import PagedLayer
from oracle import bsattn_oracle as O
from workloads import make_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build()
    B.lib()


def test_unpublished_selection_times_out_and_recovers():
    wl = make_workload(2, seed=21, T=4133)
    layer = PagedLayer(wl)
    layer.prefill()
    layer.append(0)
    torch.cuda.synchronize()
    u = next(x for x in range(wl.U) if wl.cls[x] != O.STREAMING)
    tickets = layer.workspace.view(torch.int32)[:wl.U]       # the first U words: selection tickets
    default = B.wait_limit_ns()
    B.set_wait_limit_ns(2_000_000)
    try:
        tickets[u] = 1 << 20
        layer.status.zero_()
        layer.fused_step(0)
        torch.cuda.synchronize()
        assert layer.read_status() == B.BS_ERR_TIMEOUT
    finally:
        B.set_wait_limit_ns(default)
    assert B.wait_limit_ns() == default

    # The context is still usable: zero the workspace (as the header asks after a
    # timeout), start from an empty previous selection and run the same step again.
    layer.workspace.zero_()
    layer.status.zero_()
    for i in range(2):
        layer.sel[i].fill_(-1)
        layer.cnt[i].zero_()
    layer.cur = 0
    layer.fused_step(0)
    torch.cuda.synchronize()
    assert layer.read_status() == 0
    res = O.decode_step(wl, 0, O.init_state(wl))
    got = layer.selection(0)
    out, lse = layer.out.cpu().numpy(), layer.lse.cpu().numpy()
    for v in range(wl.U):
        r = res[v]
        if not r.sel.near_tie:
            assert got[v] == r.sel.sel, v
        else:
            continue
        b, hk = divmod(v, wl.Hkv)
        o = out[b, hk * wl.G:(hk + 1) * wl.G]
        assert np.abs(o - r.o).max() <= 2e-3
        assert np.abs(lse[b, hk * wl.G:(hk + 1) * wl.G] - r.lse).max() <= 2e-3
