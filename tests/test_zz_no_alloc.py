"""spec_verify_sample_noalloc: the entry point for callers that cannot
allocate device memory (a plugin inside an engine that owns all device memory,
or a decode loop where cudaMalloc could stall other streams).  It uses a
built-in 16 MiB scratch array instead of a caller workspace.

The GPU test checks, through the C ABI, that it returns what
spec_verify_sample returns, bit for bit, and what the fp64 oracle returns,
on two calls in a row (the scratch keeps the previous call's contents, which
must not leak into the next), the first of them on a non-blocking stream.
"""
import numpy as np
import pytest

import speculative_decoding_verification_54_gb300 as sv
import workloads as wl
from speculative_decoding_verification_54_gb300 import _build


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return sv.load()


def test_noalloc_rejects_problems_beyond_its_scratch_on_host(lib):
    # B=512, gamma=31, V=262144 needs far more than 16 MiB of scratch
    A = 0x10000
    code = lib.spec_verify_sample_noalloc(A, A, sv.SPEC_BF16, A, A, A, A, 512, 31, 262144,
                                          A, A, None, None)
    assert code == sv.SPEC_ERR_WORKSPACE
    code = lib.spec_verify_sample_noalloc(None, A, sv.SPEC_BF16, A, A, A, A, 4, 4, 4096,
                                          A, A, None, None)
    assert code == sv.SPEC_ERR_INVALID_ARG
    code = lib.spec_verify_sample_noalloc(A + 8, A, sv.SPEC_BF16, A, A, A, A, 4, 4, 4096,
                                          A, A, None, None)
    assert code == sv.SPEC_ERR_ALIGNMENT


def _run_both(torch, inp, dev, stream):
    """spec_verify_sample (workspace) and spec_verify_sample_noalloc on the same
    inputs; the noalloc call goes on ``stream``."""
    from tests.gpu_util import to_device
    d = to_device(inp, dev)
    B, g, V = inp.B, inp.gamma, inp.V

    def outs():
        return (torch.full((B, g + 1), -7, dtype=torch.int32, device=dev),
                torch.full((B,), -7, dtype=torch.int32, device=dev),
                torch.zeros((B, g + 1, 4), dtype=torch.float32, device=dev))

    t0, n0, d0 = outs()
    ws = sv.make_workspace(B, g, V)
    sv.spec_verify_sample(d["target"], d["draft"], d["draft_tokens"], d["temperature"],
                          d["u_accept"], d["u_resample"], t0, n0, ws, out_debug=d0)
    assert sv.spec_verify_status(ws) == sv.SPEC_OK
    t1, n1, d1 = outs()
    torch.cuda.synchronize()  # inputs and outputs are ready before the other stream uses them
    sv.spec_verify_sample_noalloc(d["target"], d["draft"], d["draft_tokens"], d["temperature"],
                                  d["u_accept"], d["u_resample"], t1, n1, out_debug=d1, stream=stream)
    stream.synchronize()
    return [x.cpu().numpy() for x in (t0, n0, d0, t1, n1, d1)]


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_two_calls_in_a_row(lib):
    """Two calls in a row, different shapes and dtypes, the first of them the
    process's first noalloc call, on a non-blocking stream: the outputs equal
    spec_verify_sample's bit for bit (same kernels, same arithmetic) and agree
    with the fp64 oracle under the parity tests' tolerance."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import oracle
    from tests.gpu_util import assert_tally, compare
    torch.cuda.set_device(0)
    dev = torch.device("cuda:0")
    stream = torch.cuda.Stream(device=dev)  # non-blocking with respect to the legacy stream
    cases = [
        wl.make_custom(16, 4, 3 * 2048 + 40, dtype="bf16", profile="zipf", sigma=0.5,
                       temperature=("alternate", 0.0, 0.8), seed=31),
        wl.make_custom(8, 6, 8192, dtype="f32", profile="normal", sigma=0.7,
                       temperature=1.1, seed=32),
    ]
    for inp in cases:
        t0, n0, d0, t1, n1, d1 = _run_both(torch, inp, dev, stream)
        assert np.array_equal(t0, t1) and np.array_equal(n0, n1)
        assert np.array_equal(d0, d1, equal_nan=True)
        ref = oracle.verify_sample(inp.target, inp.draft, inp.draft_tokens, inp.temperature,
                                   inp.u_accept, inp.u_resample)
        assert_tally(compare(ref, t1, n1, d1))
