"""The ablation report (nvfp4_kv_cache_bd_gb300.ablation) end to end on the
GPU, on a small seeded case: every scheme packs, quantizes and decodes
through the library, and the host error budget splits the attention error
into its logit, value and probability parts.  The orderings checked are the
ones the recipe is built on: the second query term shrinks the logit error,
centering shrinks the key error, and quantizing the probabilities is the
only source of the probability part."""
import math

import numpy as np
import pytest
import torch

from nvfp4_kv_cache_bd_gb300 import ablation
import nvfp4_kv_cache_bd_gb300 as bd

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def report():
    from nvfp4_kv_cache_bd_gb300 import build
    build.build_library()
    data = ablation.Data(16 + 128 * 6 + 40, 1, 3, "cuda")
    q64 = data.q.double().cpu().numpy()
    ref = np.stack([ablation.exact_attention(q64[b], k.double().cpu().numpy(), v.double().cpu().numpy())
                    for b, (k, v) in enumerate(data.kv)])
    rows = {}
    for name, over in ablation.SCHEMES:
        if name not in ("full recipe", "one query term", "probabilities not quantized", "no key centering"):
            continue
        kw = dict(ablation.BASE, **over)
        ctx, pool, qp, gk, gv, outs = ablation.run_scheme(data, kw)
        ek, ev = ablation.key_value_errors(data, kw, pool, gk, gv)
        rl, mx = ablation.attention_errors(data, outs[1.0], ref)
        e = ablation.error_budget(data, kw, pool, qp, gk, gv, outs[1.0], ref)
        rows[name] = dict(k=ek, v=ev, rl=rl, mx=mx, **e)
        ctx.close()
    return rows


def test_every_figure_is_finite_and_consistent(report):
    for name, r in report.items():
        for key, val in r.items():
            assert math.isfinite(val), (name, key)
        # the budget's total is the report's attention error
        assert abs(r["total_rel_l2"] - r["rl"]) <= 1e-12 * max(1.0, r["rl"])
        # the three steps bound the total (triangle inequality on the same norms)
        assert r["total_rel_l2"] <= r["logits_rel_l2"] + r["values_rel_l2"] * 1.01 + r["probabilities_rel_l2"] * 1.01


def test_second_query_term_shrinks_the_logit_error(report):
    # key quantization dominates the logit error; the second term still removes a third of it here
    assert report["one query term"]["logit_rel"] > 1.2 * report["full recipe"]["logit_rel"]
    assert report["one query term"]["logits_rel_l2"] > report["full recipe"]["logits_rel_l2"]


def test_centering_shrinks_the_key_error(report):
    assert report["no key centering"]["k"] > 1.5 * report["full recipe"]["k"]


def test_probability_part_comes_from_quantizing_p(report):
    full, exact_p = report["full recipe"], report["probabilities not quantized"]
    # the same keys, values and query bytes: identical logit and value parts
    assert full["logit_rel"] == exact_p["logit_rel"] and full["values_rel_l2"] == exact_p["values_rel_l2"]
    # f16 probabilities leave a small residue; FP4 probabilities a much larger one
    assert exact_p["probabilities_rel_l2"] < full["probabilities_rel_l2"] / 3.0
