"""The assignment kernel's failure handling on the GPU, without a fault: a wait that never
completes ends with a status word and a usable device.

qvg_selftest_assign_timeout runs the tensor-core assignment with the centroid operand's load
withheld and a wait limit of one millisecond.  The kernel's MMA warp then waits on a barrier
that nothing arrives on; the bounded wait gives up, raises the kernel's abort flag and the
other roles unwind (the producer waits for the copies it issued, TMEM is freed).  The test
checks that the call returns, that QVG_DEV_TIMEOUT is set, and that a normal call afterwards
gives the bits it gave before."""
import pytest
import torch

from video_kv_cache_gb300 import api
from video_kv_cache_gb300 import build as qbuild
from video_kv_cache_gb300 import qvg, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    qbuild.build()
    qvg.load()
    torch.cuda.set_device(0)


def test_assignment_wait_gives_up_and_leaves_the_device_usable():
    X = synth.kv_tensor(51, [0, 1, 2], 0, 2, 20, 30, torch.bfloat16, "cuda")  # N = 1200
    H, N, _ = X.shape
    C, T, bits, group, iters, seed = 48, 2, 2, 32, 3, 5
    ws = api.new_workspace(H, N, C, T)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref = api.quantize(X, C, T, bits, group, iters, seed, workspace=ws, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref_bits = {k: getattr(ref, k).clone() for k in ("codes", "scales", "pi", "centroids")}

    prm = api.quant_params(H, N, C, T, bits, group, iters, X.dtype, seed)
    rc = qvg.qvg_selftest_assign_timeout(prm, X.data_ptr(), ref.buffers(), ws.data_ptr(),
                                         ws.numel(), status.data_ptr(),
                                         torch.cuda.current_stream().cuda_stream)
    assert rc == qvg.QVG_OK, qvg.qvg_status_string(rc)
    torch.cuda.synchronize()  # returns: the kernel unwound
    assert int(status.item()) & qvg.QVG_DEV_TIMEOUT

    status.zero_()
    again = api.quantize(X, C, T, bits, group, iters, seed, workspace=ws, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for k, v in ref_bits.items():
        assert torch.equal(getattr(again, k), v), k


def _small_case():
    X = synth.kv_tensor(52, [0, 1], 0, 2, 16, 24, torch.bfloat16, "cuda")  # N = 768
    H, N, _ = X.shape
    return X, H, N, 40, 2, 2, 32, 3, 9


def test_injected_launch_failure_enqueues_nothing(monkeypatch):
    """QVG_FAULT_INJECT=launch: every entry point that would enqueue device work returns
    QVG_ERR_CUDA and leaves its outputs as they were; unset, the same calls work."""
    X, H, N, C, T, bits, group, iters, seed = _small_case()
    ws = api.new_workspace(H, N, C, T)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = api.allocate(H, N, C, T, bits, group, 1, X.device)
    for k in ("codes", "scales", "pi", "centroids"):
        getattr(out, k).fill_(7)
    prm = api.quant_params(H, N, C, T, bits, group, iters, X.dtype, seed)
    stream = torch.cuda.current_stream().cuda_stream
    monkeypatch.setenv("QVG_FAULT_INJECT", "launch")
    rc = qvg.qvg_quantize(prm, X.data_ptr(), None, out.buffers(), ws.data_ptr(), ws.numel(),
                          status.data_ptr(), stream)
    assert rc == qvg.QVG_ERR_CUDA
    rc = qvg.qvg_quantize_static(prm, X.data_ptr(), None, out.buffers(), status.data_ptr(), stream)
    assert rc == qvg.QVG_ERR_CUDA
    rc = qvg.qvg_reassign(prm, X.data_ptr(), out.buffers(), ws.data_ptr(), ws.numel(),
                          status.data_ptr(), stream)
    assert rc == qvg.QVG_ERR_CUDA
    xh = torch.full((H, N, 128), 3.0, dtype=torch.float32, device="cuda")
    with pytest.raises(qvg.QVGError):
        api.dequantize(out, N, torch.float32, out=xh, status=status)
    torch.cuda.synchronize()
    for k in ("codes", "scales", "pi", "centroids"):
        assert bool((getattr(out, k) == 7).all()), k
    assert bool((xh == 3.0).all())
    assert int(status.item()) == 0
    # argument errors still come first
    bad = api.quant_params(H, N, C, T, 3, group, iters, X.dtype, seed)
    assert qvg.qvg_quantize(bad, X.data_ptr(), None, out.buffers(), ws.data_ptr(), ws.numel(),
                            None, stream) == qvg.QVG_ERR_UNSUPPORTED
    monkeypatch.delenv("QVG_FAULT_INJECT")
    rc = qvg.qvg_quantize(prm, X.data_ptr(), None, out.buffers(), ws.data_ptr(), ws.numel(),
                          status.data_ptr(), stream)
    assert rc == qvg.QVG_OK
    torch.cuda.synchronize()
    assert int(status.item()) == 0


def test_injected_alloc_failure_hits_the_static_scratch_only(monkeypatch):
    X, H, N, C, T, bits, group, iters, seed = _small_case()
    prm = api.quant_params(H, N, C, T, bits, group, iters, X.dtype, seed)
    out = api.allocate(H, N, C, T, bits, group, 1, X.device)
    stream = torch.cuda.current_stream().cuda_stream
    monkeypatch.setenv("QVG_FAULT_INJECT", "alloc")
    assert qvg.qvg_quantize_static(prm, X.data_ptr(), None, out.buffers(), None,
                                   stream) == qvg.QVG_ERR_CUDA
    ws = api.new_workspace(H, N, C, T)
    assert qvg.qvg_quantize(prm, X.data_ptr(), None, out.buffers(), ws.data_ptr(), ws.numel(),
                            None, stream) == qvg.QVG_OK
    torch.cuda.synchronize()


def test_injected_timeout_sets_the_status_and_the_next_call_is_exact(monkeypatch):
    """QVG_FAULT_INJECT=timeout: qvg_quantize's assignment waits run out (the centroid
    operand is withheld, 1 ms limit); the call returns, the status word says so, and a call
    without the injection gives the same bytes as before."""
    X, H, N, C, T, bits, group, iters, seed = _small_case()
    ws = api.new_workspace(H, N, C, T)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref = api.quantize(X, C, T, bits, group, iters, seed, workspace=ws, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref_bits = {k: getattr(ref, k).clone() for k in ("codes", "scales", "pi", "centroids")}
    monkeypatch.setenv("QVG_FAULT_INJECT", "timeout")
    api.quantize(X, C, T, bits, group, iters, seed, workspace=ws, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & qvg.QVG_DEV_TIMEOUT
    monkeypatch.delenv("QVG_FAULT_INJECT")
    status.zero_()
    again = api.quantize(X, C, T, bits, group, iters, seed, workspace=ws, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for k, v in ref_bits.items():
        assert torch.equal(getattr(again, k), v), k


def test_a_launch_failing_mid_call_enqueues_nothing_after_it(monkeypatch):
    """QVG_FAULT_INJECT=assign: the first assignment launch of qvg_quantize fails after the
    preparation kernels were enqueued.  Nothing after it may run: in particular not the
    re-scoring, whose queue no assignment wrote (the workspace is filled with 0xFF, which
    the re-scoring would report as QVG_DEV_BAD_INDEX).  The call returns QVG_ERR_CUDA, the
    status word stays clear, and a call without the injection gives the reference bytes."""
    X, H, N, C, T, bits, group, iters, seed = _small_case()
    ws = api.new_workspace(H, N, C, T)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref = api.quantize(X, C, T, bits, group, iters, seed, workspace=ws, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref_bits = {k: getattr(ref, k).clone() for k in ("codes", "scales", "pi", "centroids")}
    ws.fill_(0xFF)
    out = api.allocate(H, N, C, T, bits, group, 1, X.device)
    prm = api.quant_params(H, N, C, T, bits, group, iters, X.dtype, seed)
    stream = torch.cuda.current_stream().cuda_stream
    monkeypatch.setenv("QVG_FAULT_INJECT", "assign")
    rc = qvg.qvg_quantize(prm, X.data_ptr(), None, out.buffers(), ws.data_ptr(), ws.numel(),
                          status.data_ptr(), stream)
    assert rc == qvg.QVG_ERR_CUDA
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    monkeypatch.delenv("QVG_FAULT_INJECT")
    again = api.quantize(X, C, T, bits, group, iters, seed, workspace=ws, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for k, v in ref_bits.items():
        assert torch.equal(getattr(again, k), v), k


def test_rescoring_alone_on_an_unwritten_queue_is_skipped_and_reported():
    """qvg_reassign_steps with the re-scoring step only, on a workspace no assignment wrote
    (every byte 0xFF, so the queue's first slot and count read as -1): no request is read,
    QVG_DEV_BAD_INDEX is set, the stored assignments are untouched and the device stays
    usable."""
    X, H, N, C, T, bits, group, iters, seed = _small_case()
    ws = api.new_workspace(H, N, C, T)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = api.quantize(X, C, T, bits, group, iters, seed, workspace=ws, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    pi = out.pi.clone()
    ws.fill_(0xFF)
    api.reassign(X, out, iters, ws, seed, status=status, steps=qvg.QVG_STEP_REFINE)
    torch.cuda.synchronize()
    assert int(status.item()) & qvg.QVG_DEV_BAD_INDEX
    assert torch.equal(out.pi, pi)
    status.zero_()
    again = api.quantize(X, C, T, bits, group, iters, seed, workspace=ws, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(again.pi, pi)
