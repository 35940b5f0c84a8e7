import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300) and the built libdflash.so")
    config.addinivalue_line("markers", "slow: full-size workload check")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA GPU in this environment")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture(params=["calls", "layer", "split"])
def layer_mode(request, monkeypatch):
    """How a draft layer is issued: two calls (kv_inject, block_attn), or one
    dflash_draft_layer call with its single grouped projection launch forced on
    wherever the shapes allow it ("layer": fused per-head epilogues; "split": both
    projections as one split-K launch and one epilogue launch for both, where K allows
    two or more splits and the rows fit one row tile). Returns the run_round fused_layer
    flag."""
    if request.param in ("layer", "split"):
        monkeypatch.setenv("DFLASH_FUSED_LAYER", "1" if request.param == "layer" else "2")
        return True
    monkeypatch.delenv("DFLASH_FUSED_LAYER", raising=False)
    return False
