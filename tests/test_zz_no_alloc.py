"""The allocation-free router entry point, moe_route_topk_noalloc.

Callers whose device memory is owned by another allocator (a serving arena,
a framework plugin limited to the buffers it is handed), or whose loops must
not pay for cudaMalloc and its implicit synchronisation, cannot supply the
router's logits workspace.  This entry point keeps that scratch in a fixed
1 MiB array inside the library.  The test calls it through the C ABI and
checks it against the oracle and, bit for bit, against the workspace-taking
moe_route_topk on two calls in a row (the array keeps the first call's
contents when the second one runs), and that sizes beyond the built-in
scratch are refused with a clear error.

The file sorts last so that a run stopping at the first failure has already
run every other test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
import group_quantized_moe_gb300 as q
from group_quantized_moe_gb300 import build_lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_lib.build()
    q.lib()
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


def _with_workspace(xd, wr, bias, k):
    return q.moe_route_topk(xd, wr, bias, k)


def _noalloc_c_abi(xd, wr, bias, k):
    """Direct C-ABI call: the caller provides only inputs and outputs."""
    M, H = xd.shape
    E = wr.shape[0]
    idx = torch.empty((M, k), dtype=torch.int32, device=xd.device)
    w = torch.empty((M, k), dtype=torch.float32, device=xd.device)
    cnt = torch.empty((E,), dtype=torch.int32, device=xd.device)
    dt = q.QMM_BF16 if xd.dtype == torch.bfloat16 else q.QMM_F32
    rc = q.lib().moe_route_topk_noalloc(
        xd.data_ptr(), dt, M, H, wr.data_ptr(), None if bias is None else bias.data_ptr(), E, k,
        idx.data_ptr(), w.data_ptr(), cnt.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == q.QMM_OK, q.qmm_last_error()
    return idx, w, cnt


def _case(seed, M, E, H, k, bf16, zipf, dev):
    x = synth.normal(seed, 1, M * H).reshape(M, H)
    if bf16:
        xd = torch.from_numpy(synth.to_bf16(x).view(np.int16)).to(dev).view(torch.bfloat16)
    else:
        xd = torch.from_numpy(x).to(dev)
    wr = torch.from_numpy(synth.normal(seed, 10, E * H, 0.02).reshape(E, H)).to(dev)
    bias = torch.from_numpy(synth.zipf_bias(seed, 20, E, 1.1)).to(dev) if zipf else None
    return xd, wr, bias


def test_noalloc_router_matches_workspace_router_twice(dev):
    # Two calls in a row with different shapes and inputs: the second runs on
    # a scratch array that still holds the first call's logits.
    for seed, M, E, H, k, bf16, zipf in ((21, 512, 256, 4096, 6, True, True),
                                         (22, 8, 256, 4096, 6, False, False)):
        xd, wr, bias = _case(seed, M, E, H, k, bf16, zipf, dev)
        i0, w0, c0 = _with_workspace(xd, wr, bias, k)
        i1, w1, c1 = _noalloc_c_abi(xd, wr, bias, k)
        torch.cuda.synchronize()
        # the same kernels on the same inputs: the outputs are bit-identical,
        # so whatever the scratch held before does not leak into them
        np.testing.assert_array_equal(i1.cpu().numpy(), i0.cpu().numpy())
        np.testing.assert_array_equal(w1.cpu().numpy().view(np.uint32),
                                      w0.cpu().numpy().view(np.uint32))
        np.testing.assert_array_equal(c1.cpu().numpy(), c0.cpu().numpy())
        # and against the oracle: indices exact, weights within 2e-6
        x = xd.float().cpu().numpy()
        b = None if bias is None else bias.cpu().numpy()
        oi, ow = oracle.topk(oracle.router_logits(x, wr.cpu().numpy(), b), k)
        np.testing.assert_array_equal(i1.cpu().numpy(), oi)
        assert np.abs(w1.cpu().numpy() - ow).max() <= 2e-6
        np.testing.assert_array_equal(c1.cpu().numpy(), np.bincount(oi.reshape(-1), minlength=E))


def test_noalloc_router_at_its_scratch_limit(dev):
    # M * E equal to the built-in scratch size: the last logit of the array is
    # written and read
    E, H = 256, 64
    M = q.QMM_NOALLOC_MAX_LOGITS // E
    assert M * E == q.QMM_NOALLOC_MAX_LOGITS
    xd, wr, bias = _case(24, M, E, H, 6, False, True, dev)
    i0, w0, c0 = _with_workspace(xd, wr, bias, 6)
    i1, w1, c1 = _noalloc_c_abi(xd, wr, bias, 6)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(i1.cpu().numpy(), i0.cpu().numpy())
    np.testing.assert_array_equal(w1.cpu().numpy().view(np.uint32), w0.cpu().numpy().view(np.uint32))
    np.testing.assert_array_equal(c1.cpu().numpy(), c0.cpu().numpy())


def test_noalloc_router_refuses_sizes_beyond_its_scratch(dev):
    E, H = 256, 64
    M = q.QMM_NOALLOC_MAX_LOGITS // E + 1
    xd, wr, _ = _case(23, M, E, H, 6, False, False, dev)
    idx = torch.empty((M, 6), dtype=torch.int32, device=dev)
    w = torch.empty((M, 6), dtype=torch.float32, device=dev)
    rc = q.lib().moe_route_topk_noalloc(xd.data_ptr(), q.QMM_F32, M, H, wr.data_ptr(), None, E, 6,
                                        idx.data_ptr(), w.data_ptr(), None, None)
    assert rc == q.QMM_ERR_WORKSPACE
    assert "exceeds" in q.qmm_last_error()
    # a token count whose product with E would wrap around 64 bits is refused
    # by the same check, before anything touches the scratch
    rc = q.lib().moe_route_topk_noalloc(xd.data_ptr(), q.QMM_F32, (1 << 62) + 1, H, wr.data_ptr(),
                                        None, E, 6, idx.data_ptr(), w.data_ptr(), None, None)
    assert rc == q.QMM_ERR_WORKSPACE
