"""A numpy model of the arithmetic of libqvg's attention kernels, in fp32: the keys of a head
cut into splits of equal length (about 2048 splits over all heads, at least 64 keys and a
multiple of 32 keys each), each split walked in 32-key tiles with a running maximum and weight sum per query, and the
splits merged by rescaling to the largest maximum.  It stands in for the GPU output when the
parity checkers are themselves tested on the CPU; it is not the oracle (oracle/attention.py
is) and the library does not use it."""
import numpy as np

f32 = np.float32


def split_len(N: int, heads: int = 1) -> int:
    target = max(2048 // max(heads, 1), 1)
    length = max((N + target - 1) // target, 64)
    return (length + 31) // 32 * 32


def attention_fp32(Q, K, V, scale, heads: int = 1):
    Q, K, V = (np.asarray(a, dtype=f32) for a in (Q, K, V))
    M, N = Q.shape[0], K.shape[0]
    L = split_len(N, heads)
    S = (N + L - 1) // L
    part = np.zeros((S, M, K.shape[1]), f32)
    ml = np.zeros((S, M, 2), f32)
    for s in range(S):
        n0, n1 = s * L, min(N, s * L + L)
        mrun = np.full(M, -np.inf, f32)
        lrun = np.zeros(M, f32)
        o = np.zeros((M, K.shape[1]), f32)
        for t0 in range(n0, n1, 32):
            t1 = min(n1, t0 + 32)
            sc = (Q @ K[t0:t1].T).astype(f32) * f32(scale)
            for m in range(M):
                mnew = max(mrun[m], sc[m].max())
                corr = f32(np.exp(f32(mrun[m] - mnew)))
                p = np.exp((sc[m] - mnew).astype(f32)).astype(f32)
                lrun[m] = f32(lrun[m] * corr + p.sum(dtype=f32))
                mrun[m] = mnew
                o[m] = (o[m] * corr).astype(f32) + (p[:, None] * V[t0:t1]).sum(0, dtype=f32)
        part[s], ml[s, :, 0], ml[s, :, 1] = o, mrun, lrun
    mx = ml[:, :, 0].max(axis=0)
    w = np.exp((ml[:, :, 0] - mx).astype(f32)).astype(f32)
    l = (w * ml[:, :, 1]).sum(axis=0, dtype=f32)
    a = (w[:, :, None] * part).sum(axis=0, dtype=f32)
    return (a / l[:, None]).astype(f32)
