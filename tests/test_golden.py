"""Worked examples computed by hand (tests/golden/*.json, each with its citation and derivation):
the oracle on the CPU and the CUDA path through the C ABI must both reproduce them node by node.

The expected values are exact fractions derived on paper from the cited formulas, not outputs
of either implementation.
"""
import glob
import json
import os
from fractions import Fraction

import numpy as np
import pytest

GOLDEN = sorted(glob.glob(os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "*.json")))


def _load(path):
    with open(path) as f:
        return json.load(f)


def _val(s) -> float:
    return float(Fraction(s))


def _check(name, trees, nodes_per_tree, init_pred, pred, fx, rel):
    assert init_pred == pytest.approx(_val(fx["init_pred"]), rel=rel, abs=rel), name
    for t, want in enumerate(fx["trees"]):
        assert nodes_per_tree[t] == len(want), (name, t)
        got = trees[t][: len(want)]
        for i, w in enumerate(want):
            n = got[i]
            assert (int(n["feature"]), int(n["threshold_bin"]), int(n["left"]), int(n["right"]), int(n["is_leaf"])) == (
                w["feature"], w["threshold_bin"], w["left"], w["right"], w["is_leaf"]), (name, t, i)
            if w["is_leaf"]:
                assert float(n["leaf_value"]) == pytest.approx(_val(w["leaf_value"]), rel=rel, abs=rel), (name, t, i)
            else:
                assert float(n["gain"]) == pytest.approx(_val(w["gain"]), rel=rel), (name, t, i)
    np.testing.assert_allclose(pred, [_val(v) for v in fx["pred"]], rtol=rel, atol=rel, err_msg=name)


def test_golden_fixtures_are_cited():
    assert len(GOLDEN) >= 3
    for path in GOLDEN:
        fx = _load(path)
        assert fx["citation"] and fx["derivation"], path
        assert len(fx["bins"]) == len(fx["n_bins"]) and all(len(r) == len(fx["label"]) for r in fx["bins"])


@pytest.mark.parametrize("path", GOLDEN, ids=[os.path.basename(p)[:-5] for p in GOLDEN])
def test_oracle_matches_golden(orc, path):
    fx = _load(path)
    bins = np.array(fx["bins"], np.uint8)
    y = np.array(fx["label"], np.float32)
    out = orc.train(bins, fx["n_bins"], y, **fx["params"])
    _check(fx["name"], out["nodes"], out["nodes_per_tree"], out["init_pred"], out["pred"], fx, 1e-13)


def _cuda() -> bool:
    try:
        import torch

        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.mark.gpu
@pytest.mark.skipif(not _cuda(), reason="needs a CUDA GPU")
@pytest.mark.parametrize("path", GOLDEN, ids=[os.path.basename(p)[:-5] for p in GOLDEN])
def test_gpu_matches_golden(path):
    import torch

    import histogram_gradient_boosted_gb300 as g
    from tests.gpu_util import dev_bins

    fx = _load(path)
    bins = np.array(fx["bins"], np.uint8)
    y = np.array(fx["label"], np.float32)
    n_bins = torch.tensor(fx["n_bins"], dtype=torch.int32, device="cuda")
    out = g.train(dev_bins(bins), n_bins, torch.from_numpy(y).cuda(), **fx["params"])
    _check(fx["name"], out["nodes"], out["nodes_per_tree"], out["init_pred"], out["pred"].cpu().numpy(), fx, 1e-12)
