"""The native host pipeline (fa_host_pipeline_*, through api.HostPipeline):
steps on pinned host tensors, copies overlapped across steps, give the same
results as the direct device calls; bad arguments are rejected."""
import math

import pytest
import torch

from exact_io_aware_12_gb300 import api, _lib
from exact_io_aware_12_gb300.workloads import draw

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("depth", [1, 2, 3])
def test_pipeline_matches_direct_calls(depth):
    B, H, N, d = 1, 3, 700, 128
    steps = [draw(B, H, N, d, seed=40 + i) for i in range(4)]
    pipe = api.HostPipeline(B, H, N, d, True, depth=depth)
    hin = [{n: x[n].pin_memory() for n in ("q", "k", "v", "do")} for x in steps]
    outs = []
    for x in hin:
        o = {n: torch.empty(B, H, N, d, dtype=torch.bfloat16).pin_memory() for n in ("o", "dq", "dk", "dv")}
        o["lse"] = torch.empty(B, H, N, dtype=torch.float32).pin_memory()
        pipe.step(x["q"], x["k"], x["v"], x["do"], o["o"], o["lse"], o["dq"], o["dk"], o["dv"])
        outs.append(o)
    pipe.synchronize()
    assert api.last_device_error() == _lib.FA_OK
    for x, o in zip(steps, outs):
        q, k, v, do = (x[n].to(DEV) for n in ("q", "k", "v", "do"))
        o_ref, l_ref = api.fwd(q, k, v, True)
        dq, dk, dv = api.bwd(q, k, v, o_ref, do, l_ref, True)
        torch.cuda.synchronize()
        assert torch.equal(o["o"], o_ref.cpu()) and torch.equal(o["lse"], l_ref.cpu())
        assert torch.equal(o["dk"], dk.cpu()) and torch.equal(o["dv"], dv.cpu())
        assert (o["dq"].float() - dq.cpu().float()).abs().max().item() <= 1e-2 * max(1.0, dq.abs().max().item())


def test_pipeline_rejects_bad_arguments():
    stream = torch.cuda.current_stream().cuda_stream
    for args in [(0, 1, 128, 64, 0.1, 1, 2), (1, 1, 128, 64, 0.1, 1, 0), (1, 1, 128, 64, 0.1, 1, 9),
                 (1, 1, 128, 64, 0.0, 1, 2), (1, 1, 128, 64, 0.1, 2, 2)]:
        code, h = _lib.fa_host_pipeline_create(*args, stream)
        assert code == _lib.FA_ERR_INVALID_ARG and not h.value
    code, h = _lib.fa_host_pipeline_create(1, 1, 128, 96, 0.1, 1, 2, stream)
    assert code == _lib.FA_ERR_UNSUPPORTED
    code, h = _lib.fa_host_pipeline_create(1, 1, 128, 64, 0.1, 1, 2, stream)
    assert code == _lib.FA_OK and h.value
    assert _lib.fa_host_pipeline_step(h, None, None, None, None, None, None, None, None, None) == \
        _lib.FA_ERR_INVALID_ARG
    assert _lib.fa_host_pipeline_destroy(h) == _lib.FA_OK
    assert _lib.fa_host_pipeline_destroy(None) == _lib.FA_OK
