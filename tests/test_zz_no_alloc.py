"""qvg_quantize_static: the quantize path with the library's fixed scratch area instead of a
caller workspace.  It must give what qvg_quantize gives on the same inputs, on consecutive
calls (the second one finds the first one's leftovers in the scratch), and refuse problems
larger than the area before touching the device.

This file is named so that it is collected last: the static area is process-wide, and the
test must pass both alone and after every other test has run in the same process.
"""
import pytest
import torch

from video_kv_cache_gb300 import api
from video_kv_cache_gb300 import build as qbuild
from video_kv_cache_gb300 import qvg, synth


@pytest.fixture(scope="module")
def lib():
    qbuild.build()
    return qvg.load()


def _params(H, N, C, T, bits, group, iters, dtype, seed):
    return api.quant_params(H, N, C, T, bits, group, iters, dtype, seed)


def test_rejects_problem_larger_than_static_area(lib):
    # about 0.45 KB of scratch per token row: 200 000 rows do not fit in 64 MiB.
    prm = _params(1, 200000, 256, 2, 2, 32, 2, torch.bfloat16, 1)
    assert qvg.qvg_quantize_workspace_bytes(prm) > qvg.QVG_STATIC_SCRATCH_BYTES, "needs a larger N"
    bufs = qvg.qvg_buffers(16, 16, 16, 16)  # never dereferenced: the size check comes first
    assert qvg.qvg_quantize_static(prm, 16, None, bufs, None, None) == qvg.QVG_ERR_SCRATCH_LIMIT
    assert "qvg_quantize_static" in qvg.qvg_status_string(qvg.QVG_ERR_SCRATCH_LIMIT)
    # invalid parameters are still reported as such, not as a size problem
    bad = _params(1, 100, 256, 2, 2, 32, 2, torch.bfloat16, 1)  # C > N
    assert qvg.qvg_quantize_static(bad, 16, None, bufs, None, None) == qvg.QVG_ERR_INVALID_ARG


def _run(X, C, T, bits, group, iters, seed, static):
    H, N, _ = X.shape
    out = api.allocate(H, N, C, T, bits, group, 1, X.device)
    status = torch.zeros(1, dtype=torch.int32, device=X.device)
    prm = _params(H, N, C, T, bits, group, iters, X.dtype, seed)
    stream = torch.cuda.current_stream().cuda_stream
    if static:
        rc = qvg.qvg_quantize_static(prm, X.data_ptr(), None, out.buffers(), status.data_ptr(),
                                     stream)
    else:
        ws = api.new_workspace(H, N, C, T, X.device)
        rc = qvg.qvg_quantize(prm, X.data_ptr(), None, out.buffers(), ws.data_ptr(), ws.numel(),
                              status.data_ptr(), stream)
    assert rc == qvg.QVG_OK, qvg.qvg_status_string(rc)
    return out, status


def _assert_same(a, b, status_a, status_b):
    assert int(status_a.item()) == 0 and int(status_b.item()) == 0
    # integer outputs bit-exact; centroids compared as fp32 within zero ulp (both calls run
    # the same deterministic kernels on the same bytes)
    assert torch.equal(a.codes, b.codes)
    assert torch.equal(a.scales, b.scales)
    assert torch.equal(a.pi, b.pi)
    torch.testing.assert_close(a.centroids, b.centroids, rtol=0.0, atol=0.0)


@pytest.mark.gpu
def test_static_matches_workspace_entry_on_consecutive_calls(lib):
    torch.cuda.set_device(0)
    # two different problems back to back: 2 bf16 tensors of N = 1020 (ragged tail), T = 2,
    # INT2; then 3 fp16 tensors of N = 2040, T = 1, INT4 with 64-channel groups
    XA = synth.kv_tensor(31, [0, 1], 0, 2, 17, 30, torch.bfloat16, "cpu").cuda()
    XB = synth.kv_tensor(32, [4, 5, 6], 0, 4, 17, 30, torch.float16, "cpu").cuda()
    cfg_a = (XA, 64, 2, 2, 32, 4, 7)
    cfg_b = (XB, 100, 1, 4, 64, 3, 8)

    sa, st_sa = _run(*cfg_a, static=True)
    sb, st_sb = _run(*cfg_b, static=True)
    ra, st_ra = _run(*cfg_a, static=False)
    rb, st_rb = _run(*cfg_b, static=False)
    torch.cuda.synchronize()
    _assert_same(sa, ra, st_sa, st_ra)
    _assert_same(sb, rb, st_sb, st_rb)

    # Once set up, a repeat of the first problem takes no device memory.  Checked two ways
    # around one call: the device's free memory (cudaMemGetInfo, device-wide, so another
    # process allocating in the same window can disturb it: on a mismatch the measurement is
    # taken once more) and torch's caching-allocator counters (allocations made through this
    # process's torch).  Neither sees host memory; the header's promise of no host heap is
    # not tested here.
    torch.cuda.synchronize()
    out = api.allocate(2, XA.shape[1], 64, 2, 2, 32, 1, XA.device)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    prm = _params(2, XA.shape[1], 64, 2, 2, 32, 4, XA.dtype, 7)

    def one_call():
        torch.cuda.synchronize()
        allocs = torch.cuda.memory_stats().get("allocation.all.allocated", 0)
        free_before = torch.cuda.mem_get_info()[0]
        rc = qvg.qvg_quantize_static(prm, XA.data_ptr(), None, out.buffers(), status.data_ptr(),
                                     torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        free_after = torch.cuda.mem_get_info()[0]
        assert rc == qvg.QVG_OK
        assert torch.cuda.memory_stats().get("allocation.all.allocated", 0) == allocs
        return free_after == free_before

    assert one_call() or one_call(), "free device memory changed across two calls"
    _assert_same(out, ra, status, st_ra)
