"""Host-only checks of the C ABI: the library loads, exports every symbol include/qvg.h
declares, its struct layouts match the binding, and argument errors come back as status
codes before any device work."""
import ctypes
import os
import re
import subprocess

import pytest

from video_kv_cache_gb300 import build as qbuild
from video_kv_cache_gb300 import qvg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qvg.h")


@pytest.fixture(scope="module")
def lib():
    qbuild.build()
    return qvg.load()


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(qvg_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    declared = _declared_functions()
    assert declared == sorted(qvg.SIGNATURES), declared
    out = subprocess.run(["nm", "-D", "--defined-only", qvg.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r" T (qvg_\w+)", out))
    for name in declared:
        assert name in exported, name
        assert getattr(lib, name) is not None


def test_struct_layout_matches_header(tmp_path):
    prog = tmp_path / "layout.c"
    prog.write_text("""
#include <stddef.h>
#include <stdio.h>
#include "qvg.h"
#define F(s, f) printf("%s.%s %zu\\n", #s, #f, offsetof(s, f))
int main(void) {
  printf("qvg_quant_params %zu\\n", sizeof(qvg_quant_params));
  printf("qvg_dequant_params %zu\\n", sizeof(qvg_dequant_params));
  printf("qvg_buffers %zu\\n", sizeof(qvg_buffers));
  F(qvg_quant_params, N); F(qvg_quant_params, seed); F(qvg_quant_params, warm_stride);
  F(qvg_quant_params, table_index); F(qvg_dequant_params, chunk_len);
  F(qvg_dequant_params, out_stride); F(qvg_buffers, centroids);
  F(qvg_quant_params, qscheme); F(qvg_dequant_params, qscheme);
  F(qvg_quant_params, centroid_format);
  printf("qvg_attention_params %zu\\n", sizeof(qvg_attention_params));
  F(qvg_attention_params, N); F(qvg_attention_params, chunk_len);
  F(qvg_attention_params, scale); F(qvg_attention_params, k_first);
  F(qvg_attention_params, tensor_step);
  return 0;
}
""")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(prog), "-o", str(exe)],
                   check=True)
    got = dict(line.rsplit(" ", 1) for line in
               subprocess.run([str(exe)], capture_output=True, text=True).stdout.split("\n") if line)
    assert int(got["qvg_quant_params"]) == ctypes.sizeof(qvg.qvg_quant_params)
    assert int(got["qvg_dequant_params"]) == ctypes.sizeof(qvg.qvg_dequant_params)
    assert int(got["qvg_buffers"]) == ctypes.sizeof(qvg.qvg_buffers)
    assert int(got["qvg_attention_params"]) == ctypes.sizeof(qvg.qvg_attention_params)
    for key, st in (("qvg_quant_params", qvg.qvg_quant_params),
                    ("qvg_dequant_params", qvg.qvg_dequant_params),
                    ("qvg_buffers", qvg.qvg_buffers),
                    ("qvg_attention_params", qvg.qvg_attention_params)):
        for k, v in got.items():
            if k.startswith(key + "."):
                assert int(v) == getattr(st, k.split(".")[1]).offset, k


def _qp(**kw):
    base = dict(n_tensors=2, d=128, N=1000, C=64, T=2, bits=2, group=32, iters=3,
                in_dtype=qvg.QVG_BF16, seed=1)
    base.update(kw)
    return qvg.qvg_quant_params(**base)


def test_status_strings(lib):
    for code in range(6):
        assert qvg.qvg_status_string(code)
    assert qvg.qvg_version() == (1 << 16) | 1


def test_workspace_bytes(lib):
    a = qvg.qvg_quantize_workspace_bytes(_qp())
    b = qvg.qvg_quantize_workspace_bytes(_qp(N=2000))
    assert 0 < a < b
    # the cold-start index table grows with T
    assert qvg.qvg_quantize_workspace_bytes(_qp(T=1)) < a
    assert qvg.qvg_quantize_workspace_bytes(_qp(T=0)) <= 256
    for bad in (dict(d=64), dict(bits=3), dict(group=8), dict(C=0), dict(C=257), dict(T=9),
                dict(N=0), dict(C=1001), dict(iters=0), dict(in_dtype=7), dict(n_tensors=0)):
        assert qvg.qvg_quantize_workspace_bytes(_qp(**bad)) == 0, bad


@pytest.mark.parametrize("bad,code", [
    (dict(d=96), qvg.QVG_ERR_UNSUPPORTED), (dict(bits=8), qvg.QVG_ERR_UNSUPPORTED),
    (dict(group=128), qvg.QVG_ERR_UNSUPPORTED), (dict(T=9), qvg.QVG_ERR_UNSUPPORTED),
    (dict(C=300), qvg.QVG_ERR_UNSUPPORTED), (dict(C=200, N=100), qvg.QVG_ERR_INVALID_ARG),
    (dict(iters=0), qvg.QVG_ERR_INVALID_ARG), (dict(N=0), qvg.QVG_ERR_INVALID_ARG),
    (dict(token_offset=5), qvg.QVG_ERR_INVALID_ARG),
    (dict(token_capacity=999), qvg.QVG_ERR_INVALID_ARG),
    (dict(x_stride=128 * 999), qvg.QVG_ERR_INVALID_ARG),
    (dict(table_index=1), qvg.QVG_ERR_INVALID_ARG),
    (dict(n_tables=2, table_index=2), qvg.QVG_ERR_INVALID_ARG),
    (dict(qscheme=2), qvg.QVG_ERR_UNSUPPORTED), (dict(qscheme=-1), qvg.QVG_ERR_UNSUPPORTED),
    (dict(centroid_format=3), qvg.QVG_ERR_UNSUPPORTED),
    (dict(centroid_format=-1), qvg.QVG_ERR_UNSUPPORTED),
])
def test_quantize_rejects_bad_arguments(lib, bad, code):
    buf = (ctypes.c_ubyte * 64)()
    base = ctypes.addressof(buf) + (-ctypes.addressof(buf)) % 16
    out = qvg.qvg_buffers(base, base, base, base)
    assert qvg.qvg_quantize(_qp(**bad), base, None, out, base, 0, None, None) == code


def test_quantize_rejects_null_and_misaligned(lib):
    buf = (ctypes.c_ubyte * 64)()
    base = ctypes.addressof(buf) + (-ctypes.addressof(buf)) % 16
    good = qvg.qvg_buffers(base, base, base, base)
    assert qvg.qvg_quantize(None, base, None, good, base, 1 << 40, None, None) == qvg.QVG_ERR_INVALID_ARG
    assert qvg.qvg_quantize(_qp(), None, None, good, base, 1 << 40, None, None) == qvg.QVG_ERR_INVALID_ARG
    assert qvg.qvg_quantize(_qp(), base + 2, None, good, base, 1 << 40, None, None) == qvg.QVG_ERR_INVALID_ARG
    nopi = qvg.qvg_buffers(base, base, None, base)
    assert qvg.qvg_quantize(_qp(), base, None, nopi, base, 1 << 40, None, None) == qvg.QVG_ERR_INVALID_ARG
    # too little workspace is reported as such
    assert qvg.qvg_quantize(_qp(), base, None, good, base, 16, None, None) == qvg.QVG_ERR_WORKSPACE
    assert qvg.qvg_quantize(_qp(), base, None, good, None, 1 << 40, None, None) == qvg.QVG_ERR_WORKSPACE


def test_reassign_steps_rejects_unknown_steps(lib):
    buf = (ctypes.c_ubyte * 64)()
    base = ctypes.addressof(buf) + (-ctypes.addressof(buf)) % 16
    good = qvg.qvg_buffers(base, base, base, base)
    for steps in (8, -1, qvg.QVG_STEP_GEMM | 16):
        assert qvg.qvg_reassign_steps(_qp(), base, good, base, 1 << 40, steps, None,
                                      None) == qvg.QVG_ERR_INVALID_ARG
    # T = 0 has no assignment
    assert qvg.qvg_reassign_steps(_qp(T=0), base, good, base, 1 << 40, qvg.QVG_STEP_GEMM,
                                  None, None) == qvg.QVG_ERR_INVALID_ARG


def test_fault_injection_comes_after_the_argument_checks(lib, monkeypatch):
    # QVG_FAULT_INJECT fails calls as a launch error would, but only once their arguments
    # passed: a bad argument is still reported as such (the device is never reached here)
    buf = (ctypes.c_ubyte * 64)()
    base = ctypes.addressof(buf) + (-ctypes.addressof(buf)) % 16
    good = qvg.qvg_buffers(base, base, base, base)
    for mode in ("launch", "alloc", "timeout"):
        monkeypatch.setenv("QVG_FAULT_INJECT", mode)
        assert qvg.qvg_quantize(_qp(bits=3), base, None, good, base, 1 << 40, None,
                                None) == qvg.QVG_ERR_UNSUPPORTED
        assert qvg.qvg_quantize_static(_qp(C=5000), base, None, good, None,
                                       None) == qvg.QVG_ERR_UNSUPPORTED
        assert qvg.qvg_quantize(_qp(), base, None, good, base, 16, None,
                                None) == qvg.QVG_ERR_WORKSPACE
    # with valid arguments an injected launch failure is QVG_ERR_CUDA
    wbuf = (ctypes.c_ubyte * 512)()
    ws = ctypes.addressof(wbuf) + (-ctypes.addressof(wbuf)) % 256  # the workspace's alignment
    monkeypatch.setenv("QVG_FAULT_INJECT", "launch")
    assert qvg.qvg_quantize(_qp(), base, None, good, ws, 1 << 40, None,
                            None) == qvg.QVG_ERR_CUDA


def test_dequantize_rejects_bad_arguments(lib):
    buf = (ctypes.c_ubyte * 64)()
    base = ctypes.addressof(buf) + (-ctypes.addressof(buf)) % 16
    good = qvg.qvg_buffers(base, base, base, base)

    def dp(**kw):
        d = dict(n_tensors=1, d=128, N=100, C=16, T=1, bits=2, group=32, out_dtype=qvg.QVG_BF16)
        d.update(kw)
        return qvg.qvg_dequant_params(**d)

    for bad, code in ((dict(d=32), qvg.QVG_ERR_UNSUPPORTED), (dict(bits=1), qvg.QVG_ERR_UNSUPPORTED),
                      (dict(out_dtype=5), qvg.QVG_ERR_UNSUPPORTED), (dict(N=0), qvg.QVG_ERR_INVALID_ARG),
                      (dict(token_capacity=50), qvg.QVG_ERR_INVALID_ARG),
                      (dict(chunk_len=10, n_tables=5), qvg.QVG_ERR_INVALID_ARG),
                      (dict(out_stride=100), qvg.QVG_ERR_INVALID_ARG),
                      (dict(qscheme=3), qvg.QVG_ERR_UNSUPPORTED)):
        assert qvg.qvg_dequantize(dp(**bad), good, base, None, None) == code, bad
    assert qvg.qvg_dequantize(dp(), good, None, None, None) == qvg.QVG_ERR_INVALID_ARG
    assert qvg.qvg_dequantize(dp(), good, base + 4, None, None) == qvg.QVG_ERR_INVALID_ARG


def _ap(**kw):
    base = dict(n_heads=3, d=128, M=2, N=1000, C=64, T=2, bits=2, group=32,
                q_dtype=qvg.QVG_BF16, out_dtype=qvg.QVG_F32, scale=0.088, tensor_step=1)
    base.update(kw)
    return qvg.qvg_attention_params(**base)


def test_attention_workspace_bytes(lib):
    a = qvg.qvg_attention_workspace_bytes(_ap())
    # 16 splits of 64 keys (about 2048 over the 3 heads, at least 64 keys each), 3 heads x 2
    # queries: partial rows of 128 floats, then 2 floats each (256-byte aligned pieces)
    assert a == 3 * 16 * 2 * 128 * 4 + (3 * 16 * 2 * 2 * 4 + 255) // 256 * 256
    assert qvg.qvg_attention_workspace_bytes(_ap(M=4)) > a
    assert qvg.qvg_attention_workspace_bytes(_ap(N=100000)) > a
    for bad in (dict(M=0), dict(M=17), dict(N=0), dict(d=64), dict(bits=3), dict(group=8),
                dict(T=9), dict(C=0), dict(qscheme=2), dict(q_dtype=5), dict(out_dtype=-1),
                dict(scale=float("inf")), dict(scale=float("nan")), dict(n_heads=0),
                dict(tensor_step=-1), dict(k_first=-1), dict(token_capacity=10), dict(n_heads=65536),
                dict(chunk_len=100, n_tables=2)):
        assert qvg.qvg_attention_workspace_bytes(_ap(**bad)) == 0, bad


def test_attention_rejects_bad_arguments(lib):
    buf = (ctypes.c_ubyte * 64)()
    base = ctypes.addressof(buf) + (-ctypes.addressof(buf)) % 16
    good = qvg.qvg_buffers(base, base, base, base)
    nocent = qvg.qvg_buffers(base, base, base, None)
    big = 1 << 40
    for prm, q, kc, vc, o, ws, code in (
            (_ap(M=17), base, good, good, base, big, qvg.QVG_ERR_UNSUPPORTED),
            (_ap(N=0), base, good, good, base, big, qvg.QVG_ERR_INVALID_ARG),
            (_ap(), None, good, good, base, big, qvg.QVG_ERR_INVALID_ARG),
            (_ap(), base, good, good, None, big, qvg.QVG_ERR_INVALID_ARG),
            (_ap(), base + 2, good, good, base, big, qvg.QVG_ERR_INVALID_ARG),
            (_ap(), base, good, nocent, base, big, qvg.QVG_ERR_INVALID_ARG),
            (_ap(), base, None, good, base, big, qvg.QVG_ERR_INVALID_ARG),
            (_ap(), base, good, good, base, 16, qvg.QVG_ERR_WORKSPACE)):
        assert qvg.qvg_attention(prm, q, kc, vc, o, base, ws, None, None) == code
    assert qvg.qvg_attention(None, base, good, good, base, base, big, None, None) == \
        qvg.QVG_ERR_INVALID_ARG
    assert qvg.qvg_attention(_ap(), base, good, good, base, None, big, None, None) == \
        qvg.QVG_ERR_WORKSPACE


def test_attention_layout_defaults():
    from video_kv_cache_gb300 import api
    assert api.attention_layout(True) == (0, 1, 2)
    assert api.attention_layout(False) == (0, 0, 1)
    assert api.attention_layout(True, 4, 5, 6) == (4, 5, 6)
    assert api.attention_layout(False, v_first=3) == (0, 3, 1)


def test_static_scratch_limit_as_documented(lib):
    # about 450 B per token row plus about 630 KB per tensor, whatever T
    import torch
    from video_kv_cache_gb300 import api
    lim = qvg.QVG_STATIC_SCRATCH_BYTES

    def fits(H, N, T=2):
        return qvg.qvg_quantize_workspace_bytes(
            api.quant_params(H, N, 256, T, 2, 32, 2, torch.bfloat16, 1)) <= lim
    for T in (1, 2, 4, 8):
        assert fits(1, 145000, T) and not fits(1, 152000, T)
        assert fits(24, 4700, T) and not fits(24, 5000, T)
        assert fits(100, 240, T) and not fits(100, 270, T)
