"""The K3-shaped layer with a Zipf(s=1.1)-shaped selection bias, 16384
tokens: hot experts take many times the mean load, so the grouped GEMMs see
very ragged segments (several full 240-token tiles for one expert, many
empty experts).  Same parity contract as the uniform workloads; the bias
enters the selection key only (sigmoid(l) + b, evaluated in fp64).  The
hottest expert's first (full) work item is compared element by element, and
y on at least 256 tokens including that item's."""
import numpy as np
import pytest

import synth
from gpu_util import OracleLayer, gpu_plan, run_item_parity, run_sampled_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def zipf():
    wl = synth.workload("zipf16384")
    plan, _ = gpu_plan(wl)
    ol = OracleLayer(wl)
    yield wl, plan, ol
    plan.close()


def test_zipf16384(zipf):
    wl, plan, ol = zipf
    accepted, errs, counts, n_item = run_item_parity(wl, plan, ol, 16384)
    assert len(accepted) <= 1
    mean = 16384 * 16 / 896
    assert counts.max() > 10 * mean, f"hottest expert {counts.max()} vs mean {mean:.1f}"
    assert (counts == 0).sum() > 0
    assert n_item == 240


@pytest.mark.parametrize("T", [1, 64, 300])
def test_zipf_small_batches(zipf, T):
    """Small batches take the one-CTA-per-token top-k; with the bias every
    selection goes through the candidate band and the fp64 key ranking (and,
    above 128 tokens, the tensor-core logit estimates' band as well)."""
    wl, plan, ol = zipf
    accepted, errs, counts = run_sampled_parity(wl, plan, ol, T, np.linspace(0, T - 1, num=min(T, 24)).astype(int))
    assert len(accepted) <= 1
