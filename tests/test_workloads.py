"""The seeded input generator: determinism, shapes, bf16 rounding, page assignment."""
import numpy as np
import pytest
import torch

from workloads import DUAL, RETRIEVAL, STREAMING, bf16_bits_to_f32, make_workload, to_bf16_bits


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 10,
                        np.array([0.0, -0.0, 1.0, 1.00390625, 1.005859375, 65504.0, 3e-39], np.float32)])
    ours = to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)
    np.testing.assert_array_equal(bf16_bits_to_f32(ours),
                                  torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_deterministic_and_seed_dependent():
    a = make_workload(2, seed=3, T=2048)
    b = make_workload(2, seed=3, T=2048)
    c = make_workload(2, seed=4, T=2048)
    for name in ("K", "V", "q", "page_table"):
        np.testing.assert_array_equal(getattr(a, name), getattr(b, name))
    assert not np.array_equal(a.K, c.K)


@pytest.mark.parametrize("cfg_id,kw", [(1, {}), (2, dict(T=3000)), (3, dict(B=2, T=4000, steps=3)),
                                       (4, dict(B=3, T_range=(1000, 3000))), (5, dict(B=2, T=2000, steps=4))])
def test_shapes_and_pages(cfg_id, kw):
    wl = make_workload(cfg_id, seed=0, **kw)
    U = wl.B * wl.Hkv
    assert wl.K.shape == (U, wl.T_cap, wl.d) and wl.V.shape == wl.K.shape
    assert wl.q.shape == (wl.steps, wl.B, wl.Hq, wl.d)
    assert (wl.g % 16 == 0).all() and (wl.g % wl.s == 0).all()
    # every physical page is used by exactly one (unit, logical page)
    used = wl.page_table[wl.page_table >= 0]
    assert used.size == wl.n_pages
    np.testing.assert_array_equal(np.sort(used), np.arange(wl.n_pages))
    for u in range(U):
        n = -(-(int(wl.T_prefill[u // wl.Hkv]) + wl.steps) // 16)
        assert (wl.page_table[u, :n] >= 0).all() and (wl.page_table[u, n:] == -1).all()
    assert set(np.unique(wl.cls)) <= {STREAMING, RETRIEVAL, DUAL}
    if cfg_id == 5:
        assert wl.evict is not None and (wl.cls == DUAL).all()
    # the sink token is planted: its value norm is small against the others
    u = 0
    V = wl.V64(u)
    assert np.linalg.norm(V[0]) < 0.2 * np.linalg.norm(V[1:50], axis=1).mean()


def test_full_size_parameters_config2_and_5():
    # parameters only (cheap): k from the 5% budget and the dual budgets
    wl = make_workload(2, seed=0, T=32768)
    assert list(wl.cls) == [STREAMING] * 4 + [RETRIEVAL] * 4
    assert list(wl.k[4:]) == [51] * 4
