import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the CUDA library")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


# Backward main kernels: one CTA per key tile; the persistent kernel with one
# CTA per SM (small problems: at most one unit per CTA); the persistent kernel
# on 3 CTAs, which then take many units each.
BWD_VARIANTS = {"bwd_per_tile": (1, 0), "bwd_persistent": (2, 0), "bwd_persistent_3ctas": (2, 3)}


@pytest.fixture(params=list(BWD_VARIANTS.values()), ids=list(BWD_VARIANTS))
def bwd_variant(request):
    import scaled_dot_product_04_gb300 as m
    variant, limit = request.param
    m.sdpa_set_backward_variant(variant)
    m.sdpa_set_backward_grid_limit(limit)
    yield request.param
    m.sdpa_set_backward_variant(0)
    m.sdpa_set_backward_grid_limit(0)


# The two backward main kernels alone, each with its automatic grid (for the
# full-size workloads).
@pytest.fixture(params=[(1, 0), (2, 0)], ids=["bwd_per_tile", "bwd_persistent"])
def bwd_kernel(request):
    import scaled_dot_product_04_gb300 as m
    m.sdpa_set_backward_variant(request.param[0])
    m.sdpa_set_backward_grid_limit(request.param[1])
    yield request.param
    m.sdpa_set_backward_variant(0)
    m.sdpa_set_backward_grid_limit(0)
