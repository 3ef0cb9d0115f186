"""The ablation report's host dequantizer agrees with the test-side layout
reader (both written from the header's byte layouts) on pools the oracle
packed, and undoing rotation and centering lands near the bf16 inputs."""
import numpy as np
import pytest

import oracle
from nvfp4_kv_cache_bd_gb300 import ablation
from tests import cases, layout


@pytest.mark.parametrize("fmt", [0, 1])
def test_dequantize_pool_matches_layout_reader(fmt):
    oracle.build()
    c = cases.build(cases.Spec(lens=[16 + 128 * 3 + 5, 16 + 128 * 2], seed=5, fmt=fmt))
    pool = cases.run_oracle(c, pool_only=True)["pool"]
    pages = c.dst
    k, v = ablation.dequantize_pool(pool, fmt, pages, c.gk, c.gv)
    g_k, g_v = (c.gk, c.gv) if fmt == 0 else (1.0, 1.0)
    for i, page in enumerate(pages):
        for h in range(8):
            _, _, kv_ = layout.k_record(fmt, layout.pool_record(pool, fmt, 8, int(page), h, 0))
            _, _, vv_ = layout.v_record(fmt, layout.pool_record(pool, fmt, 8, int(page), h, 1))
            assert np.array_equal(k[i, :, h, :], kv_ * g_k)
            assert np.array_equal(v[i, :, h, :], vv_ * g_v)
    # back to the original domain: rotation undone, mean added
    kh = ablation._fwht_rows(k) + c.mu.double().numpy()
    kref = c.k_pages.double().numpy()
    assert np.linalg.norm(kh - kref) / np.linalg.norm(kref) < 0.2


def test_fwht_rows_is_its_own_inverse():
    x = np.random.default_rng(0).standard_normal((3, 5, 128))
    assert np.allclose(ablation._fwht_rows(ablation._fwht_rows(x)), x, atol=1e-12)


@pytest.mark.parametrize("fmt", [0, 1])
def test_dequantize_query_matches_layout_reader(fmt):
    """The ablation report's query dequantizer (both terms, their scales and
    g, in the rotated domain) and its q.mu field agree with the test-side
    reader on queries the oracle packed."""
    oracle.build()
    c = cases.build(cases.Spec(lens=[300, 500], seed=6, fmt=fmt))
    qp = cases.run_oracle(c, pool_only=True)["qp"]
    qh, qmu = ablation.dequantize_query(qp, fmt)
    for b in range(qp.shape[0]):
        ref_q, _, ref_mu, _, _ = layout.query_record(fmt, 32, qp[b])
        assert np.array_equal(qh[b], ref_q)
        assert np.array_equal(qmu[b], ref_mu)
