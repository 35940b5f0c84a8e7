"""dflash_ctx_project_noalloc: the context projection for callers that cannot allocate.

Callers such as a custom operator running inside another runtime's launch path
must not call cudaMalloc (that runtime owns the device memory, and allocating
would stall the device). This entry point takes its scratch from a fixed array
inside the library. The test calls it through the C ABI twice in a row, on
different inputs, and checks each result against dflash_ctx_project given an
ordinary workspace; it also checks that a call too large for the array is
refused before anything runs.
"""
import numpy as np
import pytest
import torch

import harness
from speculative_decoding_draft_dflash_gb300 import synth

pytestmark = pytest.mark.gpu


def _inputs(w, rnd, M, dt):
    counts = np.full(1, M, dtype=np.int64)
    return [torch.from_numpy(h).to("cuda", dt) for h in synth.hidden_states(w, rnd, counts)]


# f32: the walkthrough shape; bf16 at d = 4096: a block-sized call (9 K-splits), 200 rows
# (4 splits), 384 and 512 rows (2 splits), 1024 rows and 1274 rows (one split; 1274 is the
# largest that fits the array)
@pytest.mark.parametrize("name,M", [("walkthrough_f32", 3), ("qwen3_8b_b1", 128),
                                    ("qwen3_8b_b1", 200), ("qwen3_8b_b1", 384),
                                    ("qwen3_8b_b1", 512), ("qwen3_8b_b1", 1024),
                                    ("qwen3_8b_b1", 1274)])
def test_noalloc_matches_workspace_entry_point(name, M):
    from speculative_decoding_draft_dflash_gb300 import dflash as D
    w = synth.WORKLOADS[name]
    dt = torch.float32 if w.dtype == "f32" else torch.bfloat16
    dims = D.make_dims(w.d, w.n_h, w.n_kv, w.d_h, w.k, w.bs, w.eps, w.dtype)
    W_fc = torch.from_numpy(synth.W_fc(w)).to("cuda", dt)
    g_h = torch.from_numpy(synth.gamma_h(w)).to("cuda", dt)
    ws = torch.empty(D.dflash_workspace_bytes(dims, 1, 64, M), dtype=torch.uint8, device="cuda")
    for rnd in (1, 2):                       # two calls in a row, different inputs
        hid = _inputs(w, rnd, M, dt)
        ref = torch.empty((M, w.d), dtype=dt, device="cuda")
        got = torch.full((M, w.d), float("nan"), dtype=dt, device="cuda")
        D.dflash_ctx_project(dims, hid, M, W_fc, g_h, ref, ws)
        D.dflash_ctx_project_noalloc(dims, hid, M, W_fc, g_h, got)
        torch.cuda.synchronize()
        harness.check_close(got.float().cpu().numpy(), ref.float().cpu().numpy(), w.dtype,
                            f"{name} call {rnd}")
    assert D.dflash_status_get() == 0


def test_noalloc_refuses_calls_beyond_its_scratch():
    from speculative_decoding_draft_dflash_gb300 import dflash as D
    w = synth.WORKLOADS["qwen3_8b_b1"]
    dims = D.make_dims(w.d, w.n_h, w.n_kv, w.d_h, w.k, w.bs, w.eps, w.dtype)
    M = 1280                                 # one split of 1280 x 4096 fp32 + row sums > 20 MiB
    hid = [torch.zeros((M, w.d), dtype=torch.bfloat16, device="cuda") for _ in range(w.k)]
    W_fc = torch.zeros((w.d, w.k * w.d), dtype=torch.bfloat16, device="cuda")
    g_h = torch.ones(w.d, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((M, w.d), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(D.DFlashError) as e:
        D.dflash_ctx_project_noalloc(dims, hid, M, W_fc, g_h, out)
    assert e.value.status == D.ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0
