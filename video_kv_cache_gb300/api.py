"""Convenience layer over the C ABI: allocates the compressed cache and the workspace as
torch CUDA tensors and passes their pointers and the current stream to libqvg.

torch is used here only for device memory and streams; the computation is entirely in
libqvg's kernels (video_kv_cache_gb300.qvg is the ctypes binding).
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import qvg as _c

_DT = {torch.float16: _c.QVG_F16, torch.bfloat16: _c.QVG_BF16, torch.float32: _c.QVG_F32}
D = 128


@dataclass
class CompressedKV:
    """The compressed cache of H tensors (layouts as in include/qvg.h)."""
    codes: torch.Tensor      # uint8 [H][cap][d*bits/8]
    scales: torch.Tensor     # uint8 [H][cap][d/group], E4M3 bit patterns
    pi: torch.Tensor         # uint8 [H][T][cap]
    centroids: torch.Tensor  # fp32  [H][n_tables][T][C][d]
    C: int
    T: int
    bits: int
    group: int
    qscheme: int = 0         # qvg_qscheme of the codes (set by quantize)
    centroid_format: int = 0  # qvg_centroid_format of the stored centroids (set by quantize)

    @property
    def H(self):
        return self.codes.shape[0]

    @property
    def capacity(self):
        return self.codes.shape[1]

    @property
    def n_tables(self):
        return self.centroids.shape[1]

    def buffers(self) -> _c.qvg_buffers:
        return _c.qvg_buffers(self.codes.data_ptr(), self.scales.data_ptr(),
                              self.pi.data_ptr() if self.pi.numel() else None,
                              self.centroids.data_ptr() if self.centroids.numel() else None)

    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in
                   (self.codes, self.scales, self.pi, self.centroids))


def allocate(H: int, capacity: int, C: int, T: int, bits: int, group: int, n_tables: int = 1,
             device="cuda") -> CompressedKV:
    dev = torch.device(device)
    return CompressedKV(
        codes=torch.empty((H, capacity, D * bits // 8), dtype=torch.uint8, device=dev),
        scales=torch.empty((H, capacity, D // group), dtype=torch.uint8, device=dev),
        pi=torch.empty((H, T, capacity), dtype=torch.uint8, device=dev),
        centroids=torch.empty((H, n_tables, T, C if T > 0 else 0, D), dtype=torch.float32,
                              device=dev),
        C=C, T=T, bits=bits, group=group)


def quant_params(H, N, C, T, bits, group, iters, dtype, seed=0, tensor_id_base=0, x_stride=0,
                 token_offset=0, token_capacity=0, table_index=0, n_tables=0, warm_stride=0,
                 qscheme=0, centroid_format=0):
    return _c.qvg_quant_params(n_tensors=H, d=D, N=N, C=C, T=T, bits=bits, group=group,
                               iters=iters, in_dtype=_DT[dtype], seed=seed & (2 ** 64 - 1),
                               tensor_id_base=tensor_id_base, x_stride=x_stride,
                               token_offset=token_offset, token_capacity=token_capacity,
                               table_index=table_index, n_tables=n_tables,
                               warm_stride=warm_stride, qscheme=qscheme,
                               centroid_format=centroid_format)


def workspace_bytes(H: int, N: int, C: int, T: int, bits: int = 2, group: int = 32) -> int:
    return _c.qvg_quantize_workspace_bytes(
        quant_params(H, N, C, T, bits, group, 1, torch.bfloat16))


def new_workspace(H: int, N: int, C: int, T: int, device="cuda") -> torch.Tensor:
    n = workspace_bytes(H, N, C, T)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device)


def _stream_handle(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def quantize(X: torch.Tensor, C: int, T: int, bits: int, group: int, iters: int, seed: int = 0,
             *, warm: torch.Tensor | None = None, warm_stride: int = 0,
             out: CompressedKV | None = None, token_offset: int = 0, table_index: int = 0,
             workspace: torch.Tensor | None = None, status: torch.Tensor | None = None,
             tensor_id_base: int = 0, stream=None, qscheme: int = 0,
             centroid_format: int = 0) -> CompressedKV:
    """Compress X [H][N][128] (fp16 / bf16 / fp32 CUDA tensor; tensor stride may be larger
    than N*128).  With ``out`` given, writes tokens [token_offset, token_offset + N) and
    centroid table ``table_index`` of it; ``warm`` (fp32 [H][T][C][128] or a view with tensor
    stride ``warm_stride``) replaces the seeded cold start.  ``qscheme`` picks the integer
    grid of the codes (qvg.QVG_QSCHEME_*) and ``centroid_format`` the value format of the
    stored centroids (qvg.QVG_CENTROIDS_*); both are recorded in the returned cache."""
    assert X.is_cuda and X.dim() == 3 and X.shape[2] == D
    assert X.stride(2) == 1 and X.stride(1) == D
    H, N, _ = X.shape
    if out is None:
        out = allocate(H, N, C, T, bits, group, 1, X.device)
    if workspace is None:
        workspace = new_workspace(H, N, C, T, X.device)
    prm = quant_params(H, N, C, T, bits, group, iters, X.dtype, seed, tensor_id_base,
                       X.stride(0), token_offset, out.capacity, table_index, out.n_tables,
                       warm_stride, qscheme, centroid_format)
    rc = _c.qvg_quantize(prm, X.data_ptr(), warm.data_ptr() if warm is not None else None,
                         out.buffers(), workspace.data_ptr(), workspace.numel(),
                         status.data_ptr() if status is not None else None,
                         _stream_handle(stream))
    if rc != _c.QVG_OK:
        raise _c.QVGError(rc, "qvg_quantize")
    out.qscheme = qscheme
    out.centroid_format = centroid_format
    return out


def reassign(X: torch.Tensor, ckv: CompressedKV, iters: int, workspace: torch.Tensor,
             seed: int = 0, *, token_offset: int = 0, table_index: int = 0,
             status: torch.Tensor | None = None, tensor_id_base: int = 0, stream=None,
             steps: int | None = None):
    """Re-run the last stage's assignment against the stored centroids (see qvg_reassign);
    the arguments must match the preceding quantize call.  ``steps``: a mask of
    QVG_STEP_PLANES / QVG_STEP_GEMM / QVG_STEP_REFINE (qvg_reassign_steps); all by default."""
    H, N, _ = X.shape
    prm = quant_params(H, N, ckv.C, ckv.T, ckv.bits, ckv.group, iters, X.dtype, seed,
                       tensor_id_base, X.stride(0), token_offset, ckv.capacity, table_index,
                       ckv.n_tables)
    st = status.data_ptr() if status is not None else None
    if steps is None:
        rc = _c.qvg_reassign(prm, X.data_ptr(), ckv.buffers(), workspace.data_ptr(),
                             workspace.numel(), st, _stream_handle(stream))
    else:
        rc = _c.qvg_reassign_steps(prm, X.data_ptr(), ckv.buffers(), workspace.data_ptr(),
                                   workspace.numel(), steps, st, _stream_handle(stream))
    if rc != _c.QVG_OK:
        raise _c.QVGError(rc, "qvg_reassign")


def dequantize(ckv: CompressedKV, N: int | None = None, out_dtype=torch.bfloat16,
               chunk_len: int = 0, out: torch.Tensor | None = None,
               status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Reconstruct tokens [0, N) of every tensor into ``out`` [H][N][128] (tensor stride
    may be larger); token i uses centroid table i // chunk_len (0 = one table)."""
    N = ckv.capacity if N is None else N
    if out is None:
        out = torch.empty((ckv.H, N, D), dtype=out_dtype, device=ckv.codes.device)
    assert out.stride(2) == 1 and out.stride(1) == D
    prm = _c.qvg_dequant_params(n_tensors=ckv.H, d=D, N=N, C=ckv.C if ckv.T > 0 else 0, T=ckv.T,
                                bits=ckv.bits, group=ckv.group, out_dtype=_DT[out.dtype],
                                chunk_len=chunk_len, token_capacity=ckv.capacity,
                                n_tables=ckv.n_tables, out_stride=out.stride(0),
                                qscheme=ckv.qscheme)
    rc = _c.qvg_dequantize(prm, ckv.buffers(), out.data_ptr(),
                           status.data_ptr() if status is not None else None,
                           _stream_handle(stream))
    if rc != _c.QVG_OK:
        raise _c.QVGError(rc, "qvg_dequantize")
    return out


def attention_params(ckv: CompressedKV, H: int, M: int, N: int, q_dtype, out_dtype, scale: float,
                     chunk_len: int = 0, k_first: int = 0, v_first: int = 0,
                     tensor_step: int = 1):
    return _c.qvg_attention_params(
        n_heads=H, d=D, M=M, N=N, C=ckv.C if ckv.T > 0 else 0, T=ckv.T, bits=ckv.bits,
        group=ckv.group, qscheme=ckv.qscheme, chunk_len=chunk_len,
        token_capacity=ckv.capacity, n_tables=ckv.n_tables, q_dtype=_DT[q_dtype],
        out_dtype=_DT[out_dtype], scale=scale, k_first=k_first, v_first=v_first,
        tensor_step=tensor_step)


def attention_layout(one_cache: bool, k_first=None, v_first=None, tensor_step=None):
    """(k_first, v_first, tensor_step) with the defaults of ``attention`` filled in: keys and
    values interleaved in one cache (0, 1, 2), or tensor h of each of two caches (0, 0, 1)."""
    return (0 if k_first is None else k_first,
            (1 if one_cache else 0) if v_first is None else v_first,
            (2 if one_cache else 1) if tensor_step is None else tensor_step)


def attention(Q: torch.Tensor, k_cache: CompressedKV, v_cache: CompressedKV | None = None,
              scale: float | None = None, N: int | None = None, *, out_dtype=torch.float32,
              chunk_len: int = 0, k_first: int | None = None, v_first: int | None = None,
              tensor_step: int | None = None, out: torch.Tensor | None = None,
              workspace: torch.Tensor | None = None, status: torch.Tensor | None = None,
              stream=None) -> torch.Tensor:
    """Softmax attention of Q [H][M][128] over tokens [0, N) of compressed keys and values
    (qvg_attention): head h reads key tensor k_first + h * tensor_step of ``k_cache`` and
    value tensor v_first + h * tensor_step of ``v_cache``.  With one cache (``v_cache``
    omitted) the default layout is keys and values interleaved, tensors 2h and 2h + 1; with
    two caches it is tensor h of each.  ``scale`` defaults to 1 / sqrt(128)."""
    k_first, v_first, tensor_step = attention_layout(v_cache is None, k_first, v_first,
                                                     tensor_step)
    v_cache = k_cache if v_cache is None else v_cache
    assert Q.is_cuda and Q.dim() == 3 and Q.shape[2] == D and Q.is_contiguous()
    H, M, _ = Q.shape
    N = k_cache.capacity if N is None else N
    scale = D ** -0.5 if scale is None else scale
    if out is None:
        out = torch.empty((H, M, D), dtype=out_dtype, device=Q.device)
    assert out.is_contiguous() and out.shape == (H, M, D)
    prm = attention_params(k_cache, H, M, N, Q.dtype, out.dtype, scale, chunk_len, k_first,
                           v_first, tensor_step)
    need = _c.qvg_attention_workspace_bytes(prm)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=Q.device)
    rc = _c.qvg_attention(prm, Q.data_ptr(), k_cache.buffers(), v_cache.buffers(),
                          out.data_ptr(), workspace.data_ptr(), workspace.numel(),
                          status.data_ptr() if status is not None else None,
                          _stream_handle(stream))
    if rc != _c.QVG_OK:
        raise _c.QVGError(rc, "qvg_attention")
    return out
