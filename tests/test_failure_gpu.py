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
