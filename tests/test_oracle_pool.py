"""The process-parallel oracle helper used by the full-size GPU tests gives
exactly what the plain oracle calls give (CPU only)."""
import numpy as np
import pytest

import oracle
from tests import cases
from tests.fullsize import OraclePool


@pytest.fixture(scope="module")
def opool():
    oracle.build()
    p = OraclePool(procs=2)
    yield p
    p.close()


def test_parallel_writer_and_decode_equal_the_plain_oracle(opool):
    c = cases.build(cases.Spec(lens=[16 + 128 * 5 + 7, 300, 16 + 128 * 3], seed=11))
    ref = cases.run_oracle(c)
    kw = dict(fmt=0, key_search=1, rotation=1, centering=1, query_terms=2, p_mode=2, p_c=8)
    pool = np.full_like(ref["pool"], cases.FILL)
    opool.quantize_pages(kw, cases.u16(c.k_pages), cases.u16(c.v_pages), c.dst, c.mu.numpy(), c.gk, c.gv, pool)
    assert np.array_equal(pool, ref["pool"])
    out = opool.decode(kw, ref["qp"], cases.u16(c.q), c.mu.numpy(), pool, c.block_table, c.seq_lens,
                       cases.u16(c.sink_k), cases.u16(c.sink_v), cases.u16(c.tail_k), cases.u16(c.tail_v),
                       c.spec.tau, c.gk, c.gv)
    assert np.array_equal(out, ref["out"])
