"""cp_frame_static: the frame with its working set in the library's static
scratch array instead of memory the handle allocated.

It serves callers that cannot allocate device memory where they run a frame
(inside an open stream capture, under an allocator that owns the device, on a
thread that must not block in cudaMalloc). The test runs it twice in a row
through the C ABI and checks both calls against cp_frame on the same inputs
(the same tiles in the same order, so the results are bit-identical, which is
within every tolerance the other tests use), checks the size limit where the
header states it, and checks that its device-side errors reach cp_status.

This file sorts last so that a run stopping at its first failure has already
run every other test; it also passes when run alone in a fresh process.
"""
import numpy as np
import pytest
import torch

import helpers
from persistent_megakernel_streaming_gb300 import cp, torch_io

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _run(fn, s, h, c0, samp_np):
    R, P = h.shape[0], s["positions"]
    ts = torch_io.sampler_to_torch(samp_np)
    codes = torch.full((R, P - 1), -1, dtype=torch.int32, device="cuda")
    es = torch.zeros((R, s["hidden"]), dtype=torch.float32, device="cuda")
    fn(torch.from_numpy(h).cuda(), torch.from_numpy(c0).cuda(), ts, R, codes, es)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), es.cpu().numpy(), ts["offset"].cpu().numpy()


@pytest.mark.parametrize("name,rows", [("tiny", 64), ("full", 16), ("full_r128", 20)])
def test_static_scratch_frame_matches_cp_frame_twice(name, rows):
    fr = helpers.handle(name)
    s = fr.shape
    h, c0, samp = helpers.inputs(name, rows, "mixed", seed=11)
    want = _run(fr.frame, s, h, c0, samp)
    assert fr.status() == 0
    for call in range(2):
        got = _run(fr.frame_static, s, h, c0, samp)
        for a, b, what in zip(want, got, ("codes", "emb_sum", "offset")):
            np.testing.assert_array_equal(a, b, err_msg=f"call {call}: {what}")
    assert (want[0] >= 0).all()


# the most rows whose working set fits the static array at the 1.7B shape
# (the header states it: 25 rows take 16.64 MB of the 16 MiB, 26 take 16.88 MB)
STATIC_MAX_ROWS_FULL = 25


def test_static_scratch_limit_is_where_the_header_says():
    """The last row count that fits runs and matches cp_frame bit for bit; one
    more row, and 64, are refused with CP_ERR_SCRATCH_LIMIT before anything
    is launched."""
    fr = helpers.handle("full")
    s = fr.shape
    R = STATIC_MAX_ROWS_FULL
    h, c0, samp = helpers.inputs("full", R, "mixed", seed=13)
    want = _run(fr.frame, s, h, c0, samp)
    got = _run(fr.frame_static, s, h, c0, samp)
    for a, b, what in zip(want, got, ("codes", "emb_sum", "offset")):
        np.testing.assert_array_equal(a, b, err_msg=what)
    for rows in (R + 1, 64):
        h, c0, samp = helpers.inputs("full", rows, "greedy", seed=0)
        with pytest.raises(cp.CPError) as e:
            _run(fr.frame_static, s, h, c0, samp)
        assert e.value.code == cp.CP_ERR_SCRATCH_LIMIT


def test_static_scratch_errors_reach_cp_status():
    """A device-side error of this call is the handle's sticky status, as for
    cp_frame: a wait that nothing satisfies ends the call with CP_ERR_TIMEOUT
    after the handle's limit, cp_status reports it, further calls return at
    once until it is cleared, and cleared, the handle's status is CP_OK."""
    fr = helpers.handle("tiny", debug_stall_task=3, timeout_ns=50_000_000)
    s = fr.shape
    h, c0, samp = helpers.inputs("tiny", 2, "greedy", seed=0)
    _run(fr.frame_static, s, h, c0, samp)
    assert fr.status() == cp.CP_ERR_TIMEOUT
    _run(fr.frame_static, s, h, c0, samp)   # skipped: the status is sticky
    assert fr.status() == cp.CP_ERR_TIMEOUT
    fr.clear_status()
    assert fr.status() == 0
