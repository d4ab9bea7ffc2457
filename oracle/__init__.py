"""CPU oracle for frame-aligned window-sparse attention.

TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
cpu_baseline / reference legs of bench.py may import this package.  It shares
no code with the CUDA library (frame_aligned_window_gb300) and never imports
it; the only module both sides use is `workloads` (seeded inputs).

`oracle.c` is plain fp64 C (built here with gcc and OpenMP); `produce` (the
pre-attention producer) is numpy in fp64 with a library matmul; `brute.py` is
a second, pure-Python restatement used to pin both on tiny inputs.

Parity status: every function here is pinned by tests under tests/ against
brute force, closed forms, invariants or a library routine (see the
test_oracle_* files).  The pages' TPU figures (fraction of the TPU bound,
share of eligible heads) are context only and not pinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lib = None
_lock = threading.Lock()

# tau of the fixed-max eligibility test, in scaled-logit units (the library's
# constant; the pages give no value).
TAU = 40.0


def build(force: bool = False) -> str:
    """Compiles oracle.c into _build/liboracle.so with gcc -O2 -fopenmp."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            L, P, D = ctypes.c_long, ctypes.c_void_p, ctypes.c_double
            lib.orc_mask.argtypes = [L, L, L, L, L, L, L]
            lib.orc_mask.restype = ctypes.c_int
            lib.orc_mask_dense.argtypes = [L, L, L, L, L, P]
            lib.orc_blockmap.argtypes = [L, L, L, L, L, L, L, P, P, P, L, P]
            lib.orc_blockmap.restype = ctypes.c_int
            lib.orc_prepare.argtypes = [P, P, L, L, L, D, D, P, P, P, P, P, P]
            lib.orc_prepare_window.argtypes = [P, P, L, L, L, L, L, L, L, L, D, D, P, P, P,
                                               P, P, P]
            lib.orc_attention_rows.argtypes = [P, P, P, L, L, L, L, L, L, L, D, L, P, P, P]
            lib.orc_attention_rows_fixed.argtypes = [P, P, P, P, P, L, L, L, L, L, L, L, D, L,
                                                     P, P, P]
            lib.orc_attention_rows_online.argtypes = [P, P, P, L, L, L, L, L, L, L, D, L, L, P,
                                                      P, P]
            lib.orc_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def num_threads() -> int:
    return int(_load().orc_num_threads())


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def as_f64(x) -> np.ndarray:
    """[..., N, D] bf16/float tensor or array -> contiguous float64 [nbh, N, D]
    (exact for bf16 and fp32 inputs)."""
    if isinstance(x, torch.Tensor):
        x = x.detach().to("cpu").to(torch.float64).numpy()
    x = np.ascontiguousarray(x, dtype=np.float64)
    return x.reshape(-1, x.shape[-2], x.shape[-1])


# Mask variants (or-ed; 0 = symmetric window, reference frames first,
# reference queries global): see orc_mask.
MASK_CAUSAL = 1
MASK_REF_SUFFIX = 2
MASK_REF_LOCAL = 4


def mask(F, T, w, R, i, j, flags: int = 0) -> int:
    return int(_load().orc_mask(F, T, w, R, flags, i, j))


def mask_dense(F, T, w, R, flags: int = 0) -> np.ndarray:
    n = (F + R) * T
    out = np.zeros((n, n), dtype=np.uint8)
    _load().orc_mask_dense(F, T, w, R, flags, _ptr(out))
    return out


def blockmap(F, T, w, R, bq, bk, flags: int = 0) -> dict:
    n = (F + R) * T
    if bq <= 0 or bk <= 0 or n % bq or n % bk:
        raise ValueError("block sizes must tile the sequence")
    nqb, nkb = n // bq, n // bk
    bitmap = np.zeros(nqb * nkb, dtype=np.uint8)
    row_ptr = np.zeros(nqb + 1, dtype=np.int32)
    col = np.zeros(nqb * nkb, dtype=np.int32)
    counts = np.zeros(4, dtype=np.int64)
    rc = _load().orc_blockmap(F, T, w, R, flags, bq, bk, _ptr(bitmap), _ptr(row_ptr),
                              _ptr(col), nqb * nkb, _ptr(counts))
    if rc != 0:
        raise RuntimeError("orc_blockmap failed")
    nnz = int(counts[3])
    return {"bitmap": bitmap.reshape(nqb, nkb), "row_ptr": row_ptr, "col": col[:nnz].copy(),
            "full": int(counts[0]), "empty": int(counts[1]), "partial": int(counts[2]),
            "nnz": nnz}


def prepare(q, k, scale: float, tau: float = TAU) -> dict:
    """fp64 per-head statistics; q, k are [..., N, D]."""
    qd, kd = as_f64(q), as_f64(k)
    nbh, n, d = kd.shape
    mu = np.zeros((nbh, d)); kmax = np.zeros(nbh); qn = np.zeros((nbh, n))
    b = np.zeros((nbh, n)); bmax = np.zeros(nbh); elig = np.zeros(nbh, dtype=np.uint8)
    _load().orc_prepare(_ptr(qd), _ptr(kd), nbh, n, d, scale, tau, _ptr(mu), _ptr(kmax),
                        _ptr(qn), _ptr(b), _ptr(bmax), _ptr(elig))
    return {"mu": mu, "kmax": kmax, "qn": qn, "b": b, "bmax": bmax, "elig": elig}


def prepare_window(q, k, F, T, w, R, scale: float, tau: float = TAU, flags: int = 0) -> dict:
    """Like prepare(), with each row's bound over the keys its row attends
    (the mask walked element by element).  kmax stays the global maximum."""
    qd, kd = as_f64(q), as_f64(k)
    nbh, n, d = kd.shape
    mu = np.zeros((nbh, d)); kmax = np.zeros(nbh); qn = np.zeros((nbh, n))
    b = np.zeros((nbh, n)); bmax = np.zeros(nbh); elig = np.zeros(nbh, dtype=np.uint8)
    _load().orc_prepare_window(_ptr(qd), _ptr(kd), nbh, n, d, F, T, w, R, flags, scale, tau,
                               _ptr(mu), _ptr(kmax), _ptr(qn), _ptr(b), _ptr(bmax), _ptr(elig))
    return {"mu": mu, "kmax": kmax, "qn": qn, "b": b, "bmax": bmax, "elig": elig}


def _pairs(pairs):
    p = np.asarray(pairs, dtype=np.int64).reshape(-1, 2)
    return np.ascontiguousarray(p[:, 0]), np.ascontiguousarray(p[:, 1])


def attention_rows(q, k, v, F, T, w, R, scale, pairs, flags: int = 0) -> np.ndarray:
    """Plain masked softmax attention for (head, row) pairs -> [npairs, D].
    Heads index the flattened [nbh] axis of q, k, v."""
    qd, kd, vd = as_f64(q), as_f64(k), as_f64(v)
    nbh, n, d = kd.shape
    h, r = _pairs(pairs)
    out = np.zeros((len(h), d))
    _load().orc_attention_rows(_ptr(qd), _ptr(kd), _ptr(vd), n, d, F, T, w, R, flags, scale,
                               len(h), _ptr(h), _ptr(r), _ptr(out))
    return out


def attention_rows_fixed(q, k, v, F, T, w, R, scale, pairs, stats, flags: int = 0) -> np.ndarray:
    qd, kd, vd = as_f64(q), as_f64(k), as_f64(v)
    nbh, n, d = kd.shape
    h, r = _pairs(pairs)
    mu = np.ascontiguousarray(stats["mu"], dtype=np.float64)
    b = np.ascontiguousarray(stats["b"], dtype=np.float64)
    out = np.zeros((len(h), d))
    _load().orc_attention_rows_fixed(_ptr(qd), _ptr(kd), _ptr(vd), _ptr(mu), _ptr(b), n, d, F,
                                     T, w, R, flags, scale, len(h), _ptr(h), _ptr(r), _ptr(out))
    return out


def attention_rows_online(q, k, v, F, T, w, R, scale, bk, pairs, flags: int = 0) -> np.ndarray:
    qd, kd, vd = as_f64(q), as_f64(k), as_f64(v)
    nbh, n, d = kd.shape
    h, r = _pairs(pairs)
    out = np.zeros((len(h), d))
    _load().orc_attention_rows_online(_ptr(qd), _ptr(kd), _ptr(vd), n, d, F, T, w, R, flags,
                                      scale, bk, len(h), _ptr(h), _ptr(r), _ptr(out))
    return out


def attention_full(q, k, v, F, T, w, R, scale, flags: int = 0) -> np.ndarray:
    """Every row of every head: [nbh, N, D] (small shapes)."""
    kd = as_f64(k)
    nbh, n, d = kd.shape
    pairs = [(h, i) for h in range(nbh) for i in range(n)]
    return attention_rows(q, k, v, F, T, w, R, scale, pairs, flags).reshape(nbh, n, d)


def produce(x, w, rope_cos, rope_sin, eps: float, heads: int, head_dim: int, rows=None):
    """Pre-attention producer, plain definition in fp64 -> (q, k, v).

    Google Developers Blog post "HeyGen x Google Cloud: Bringing Avatar IV to
    TPUs", section "Layout is ABI" and Figure 5: a chain of small ops
    (normalisation, rotary embedding, projection, head packing) produces the
    attention inputs, and one fused kernel writes them straight into the
    layout the consumer reads.  The pages name the ops only; this oracle takes
    the plainest reading of each:

      1. RMS normalisation of every token, without a gain (a gain is folded
         into the projection weights by the caller):
         xh_t = x_t / sqrt(mean_c x_tc^2 + eps);
      2. projection without bias: y_t = W xh_t, W [3 H D, C] whose rows are
         the q features (head-major, dim-minor), then k, then v;
      3. rotary embedding of q and k: dims (2p, 2p+1) of token t turn by the
         angle whose cosine and sine are rope_cos[t, p], rope_sin[t, p]
         ((a, b) -> (a cos - b sin, a sin + b cos)); v is not rotated;
      4. head packing into [B, H, N, D].

    x: [B, N, C]; w: [3 H D, C]; rope_cos, rope_sin: [N, D / 2] (the table is
    an input: it encodes the positions).  rows: token indices to compute
    (default all).  Returns three float64 arrays [B, H, len(rows), D].
    """
    xd = np.asarray(x.detach().cpu().to(torch.float64).numpy() if isinstance(x, torch.Tensor)
                    else x, dtype=np.float64)
    wd = np.asarray(w.detach().cpu().to(torch.float64).numpy() if isinstance(w, torch.Tensor)
                    else w, dtype=np.float64)
    cd = np.asarray(rope_cos.detach().cpu().to(torch.float64).numpy()
                    if isinstance(rope_cos, torch.Tensor) else rope_cos, dtype=np.float64)
    sd = np.asarray(rope_sin.detach().cpu().to(torch.float64).numpy()
                    if isinstance(rope_sin, torch.Tensor) else rope_sin, dtype=np.float64)
    B, N, C = xd.shape
    H, D = heads, head_dim
    if wd.shape != (3 * H * D, C) or cd.shape != (N, D // 2) or sd.shape != (N, D // 2):
        raise ValueError("produce: shape mismatch")
    rows = np.arange(N) if rows is None else np.asarray(rows, dtype=np.int64)
    xs = xd[:, rows, :]                                            # [B, n, C]
    xh = xs / np.sqrt(np.mean(xs * xs, axis=2, keepdims=True) + eps)
    y = xh @ wd.T                                                  # [B, n, 3 H D]
    y = y.reshape(B, len(rows), 3, H, D)
    c = cd[rows][None, :, None, :]                                 # [1, n, 1, D/2]
    s = sd[rows][None, :, None, :]

    def rotate(t):
        a, b = t[..., 0::2], t[..., 1::2]
        out = np.empty_like(t)
        out[..., 0::2] = a * c - b * s
        out[..., 1::2] = a * s + b * c
        return out

    q = rotate(y[:, :, 0])
    k = rotate(y[:, :, 1])
    v = y[:, :, 2]
    pack = lambda t: np.ascontiguousarray(t.transpose(0, 2, 1, 3))  # noqa: E731
    return pack(q), pack(k), pack(v)
