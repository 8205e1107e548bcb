"""The attention entry point that needs no workspace from its caller.

It serves callers that cannot allocate device memory, such as a plugin whose host
engine owns all allocations, or a serving loop that must not call cudaMalloc after
start-up. The test drives it through the C ABI and checks two calls in a row against
bs_sparse_decode_attn with a caller-allocated workspace and against the float64
oracle's attention over the same selections, and that a shape too large for its fixed
scratch array is refused on the host. It lives in a file of its own so that pytest
collects it last.
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

ATT_ABS, ATT_REL, REL_FLOOR = 2e-3, 1e-2, 0.2


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build()
    B.lib()


def _close(a, ref):
    diff = (a.double() - ref.double()).abs()
    assert float(diff.max()) <= ATT_ABS
    assert float((diff / ref.double().abs().clamp_min(REL_FLOOR)).max()) <= ATT_REL


@pytest.mark.parametrize("large", [False, True], ids=["cluster-merge", "scratch-merge"])
def test_noalloc_matches_workspace_entry_point_on_two_calls(large):
    """Small selections merge their splits on chip; selections above 1024 pages keep
    their split partials in the fixed scratch array."""
    wl = make_workload(2, seed=11, T=20000 if large else 5000)
    if large:
        wl.k[4:] = 600                  # ~1200 pages per retrieval unit
    layer = PagedLayer(wl)
    layer.prefill()
    layer.append(0)
    layer.update_summaries(0)
    layer.score(0)
    layer.select(0)
    layer.attend(0)                     # caller-allocated workspace
    torch.cuda.synchronize()
    ref_out, ref_lse = layer.out.clone(), layer.lse.clone()
    assert layer.read_status() == 0
    # The float64 oracle's attention over the selections the GPU made.
    sel = layer.selection(layer.cur)
    oracle_out = np.zeros(tuple(layer.out.shape))
    oracle_lse = np.zeros(tuple(layer.lse.shape))
    for u in range(wl.U):
        b, hk = divmod(u, wl.Hkv)
        o, lse = O.sparse_attention(wl.q64(0, u), wl.K64(u), wl.V64(u), sel[u], int(wl.g[u]), wl.T(0, b))
        oracle_out[b, hk * wl.G:(hk + 1) * wl.G] = o
        oracle_lse[b, hk * wl.G:(hk + 1) * wl.G] = lse
    for _ in range(2):
        layer.out.fill_(float("nan"))
        layer.lse.fill_(float("nan"))
        B.sparse_decode_attn_noalloc(layer.dims, layer.q[0], layer.kv_at(layer.seq_lens[0]), layer.cfg,
                                     layer.sel[layer.cur], layer.cnt[layer.cur], layer.out, layer.lse,
                                     layer.status)
        torch.cuda.synchronize()
        assert layer.read_status() == 0
        _close(layer.out, ref_out)
        _close(layer.lse, ref_lse)
        _close(layer.out, torch.from_numpy(oracle_out).to(layer.out.device))
        assert float((layer.lse.double().cpu() - torch.from_numpy(oracle_lse)).abs().max()) <= ATT_ABS


def test_noalloc_refuses_dims_beyond_its_scratch():
    wl = make_workload(2, seed=12, T=3000)
    layer = PagedLayer(wl)
    big = B.Dims.from_buffer_copy(layer.dims)
    big.batch = 64                        # 512 units
    big.max_gather_pages_per_unit = 4000  # page lists alone take 8.2 MB
    assert B.workspace_size(big) > 8 << 20
    status = B.lib().bs_sparse_decode_attn_noalloc(
        B.ctypes.byref(big), layer.q[0].data_ptr(), B.ctypes.byref(layer.kv_at(layer.seq_lens[0])),
        B.ctypes.byref(layer.cfg), layer.sel[0].data_ptr(), layer.cnt[0].data_ptr(), None, layer.out.data_ptr(),
        layer.lse.data_ptr(), layer.status.data_ptr(), None)
    assert status == B.BS_ERR_CAPACITY
