"""Python binding of libwsattn (frame-aligned window-sparse attention, GB300).

Argument marshalling only: every step of the computation runs in the CUDA
library (include/wsattn.h documents each call).  Tensors are torch tensors
used as device memory; the current torch CUDA stream is passed to the
library.  If libwsattn.so is missing or fails to load, importing this
package raises: there is no fallback implementation.  The environment
variable WSATTN_LIBRARY names another build of the same library to load
instead (the tests use it for the bounds-checking libwsattn_debug.so).

The names mirror the C ABI:
    wsattn_plan, wsattn_plan_ex, wsattn_plan_destroy, wsattn_prepare, wsattn_forward,
    wsattn_plan_info, wsattn_get_tiles, wsattn_get_block_map, wsattn_get_csr, wsattn_get_stats,
    wsattn_plan_set_debug, wsattn_plan_set_bound, wsattn_device_status,
    wsattn_selftest_timeout, wsattn_status_string, wsattn_prepare_static, wsattn_produce,
    wsattn_build_flags
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.environ.get("WSATTN_LIBRARY") or os.path.join(_HERE, "libwsattn.so")
DEBUG_LIB_PATH = os.path.join(_HERE, "libwsattn_debug.so")

# C ABI entry points declared in include/wsattn.h
EXPORTS = (
    "wsattn_plan", "wsattn_plan_ex", "wsattn_plan_destroy", "wsattn_prepare", "wsattn_forward",
    "wsattn_plan_info", "wsattn_get_tiles", "wsattn_get_block_map", "wsattn_get_csr",
    "wsattn_get_stats",
    "wsattn_plan_set_debug", "wsattn_plan_set_bound", "wsattn_device_status",
    "wsattn_selftest_timeout", "wsattn_status_string", "wsattn_prepare_static",
    "wsattn_produce", "wsattn_build_flags",
)

# wsattn_bound
BOUND_GLOBAL = 0
BOUND_WINDOW = 1

# wsattn_mask_flags (or-ed)
MASK_CAUSAL = 1
MASK_REF_SUFFIX = 2
MASK_REF_LOCAL = 4

STATUS = {0: "OK", 1: "BAD_ARG", 2: "BAD_BLOCK", 3: "UNSUPPORTED", 4: "NOT_PREPARED",
          5: "BATCH_MISMATCH", 6: "CUDA", 7: "TIMEOUT", 8: "NO_MEMORY", 9: "BOUNDS"}

# wsattn_build_flags bits
BUILD_DEBUG = 1


class WsattnError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {STATUS.get(code, code)} ({status_text(code)})")


if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with "
                      "`python frame_aligned_window_gb300/build.py`"
                      + (" --debug" if LIB_PATH == DEBUG_LIB_PATH else ""))
_lib = ctypes.CDLL(LIB_PATH)

_P, _I, _F, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
_lib.wsattn_plan.argtypes = [_I, _I, _I, _I, _I, _I, _I, _I, ctypes.POINTER(_P)]
_lib.wsattn_plan_ex.argtypes = [_I, _I, _I, _I, _I, _I, _I, _I, _I, ctypes.POINTER(_P)]
_lib.wsattn_plan_destroy.argtypes = [_P]
_lib.wsattn_prepare.argtypes = [_P, _I, _P, _P, _P]
_lib.wsattn_forward.argtypes = [_P, _I, _P, _P, _P, _P, _P]
_lib.wsattn_plan_info.argtypes = [_P, _P, _I]
_lib.wsattn_get_block_map.argtypes = [_P, _P, _SZ]
_lib.wsattn_get_csr.argtypes = [_P, _P, _P, _SZ, _SZ]
_lib.wsattn_get_tiles.argtypes = [_P, _P, _SZ, _P, _SZ]
_lib.wsattn_get_stats.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P]
_lib.wsattn_plan_set_debug.argtypes = [_P, _I, _F]
_lib.wsattn_plan_set_bound.argtypes = [_P, _I]
_lib.wsattn_device_status.argtypes = [_P, _P]
_lib.wsattn_selftest_timeout.argtypes = [_I, ctypes.POINTER(_I), _P]
_lib.wsattn_status_string.argtypes = [_I]
_lib.wsattn_prepare_static.argtypes = [_I, _I, _I, _I, _F, _P, _P, _P, _P, _P, _P, _P, _P, _P]
_lib.wsattn_produce.argtypes = [_P, _I, _P, _I, _P, _P, _P, _F, _P, _P, _P, _P]
_lib.wsattn_build_flags.argtypes = []
_lib.wsattn_status_string.restype = ctypes.c_char_p
for _name in EXPORTS:
    if _name != "wsattn_status_string":
        getattr(_lib, _name).restype = _I


def wsattn_build_flags() -> int:
    """BUILD_DEBUG when the loaded library checks bounds in its kernels."""
    return int(_lib.wsattn_build_flags())


def status_text(code: int) -> str:
    return _lib.wsattn_status_string(int(code)).decode()


def wsattn_status_string(code: int) -> str:
    return status_text(code)


def _check(rc: int, what: str):
    if rc != 0:
        raise WsattnError(rc, what)


class Plan:
    """Owns a wsattn_plan_t handle (released by destroy() or on collection)."""

    def __init__(self, handle, args):
        self._h = handle
        self.args = args
        info = np.zeros(10, dtype=np.int64)
        _check(_lib.wsattn_plan_info(self._h, info.ctypes.data, 10), "wsattn_plan_info")
        (self.n_tokens, self.block_q, self.block_k, self.n_qblocks, self.n_kblocks, self.nnz,
         self.tiles_per_head, self.head_dim, self.heads, self.active_pairs) = (int(x) for x in info)
        self.frames, self.tokens_per_frame, self.window, self.ref_frames = args[:4]

    @property
    def handle(self):
        if self._h is None:
            raise ValueError("plan was destroyed")
        return self._h

    def destroy(self):
        if self._h is not None:
            _lib.wsattn_plan_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


def _stream_ptr(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dev_ptr(t, name, dtype=None):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _check_shape(plan: Plan, t, name):
    if t.dim() != 4 or t.shape[1] != plan.heads or t.shape[2] != plan.n_tokens \
            or t.shape[3] != plan.head_dim:
        raise ValueError(f"{name} must be [B, {plan.heads}, {plan.n_tokens}, {plan.head_dim}], "
                         f"got {tuple(t.shape)}")


def wsattn_plan(frames, tokens_per_frame, window, ref_frames, heads, head_dim, block_q=0,
                block_k=0, mask_flags=0) -> Plan:
    """wsattn_plan_ex when mask_flags != 0 (MASK_* or-ed), else wsattn_plan."""
    h = _P()
    args = (frames, tokens_per_frame, window, ref_frames, heads, head_dim, block_q, block_k)
    if mask_flags:
        _check(_lib.wsattn_plan_ex(*args, int(mask_flags), ctypes.byref(h)), "wsattn_plan_ex")
    else:
        _check(_lib.wsattn_plan(*args, ctypes.byref(h)), "wsattn_plan")
    plan = Plan(h, args)
    plan.mask_flags = int(mask_flags)
    return plan


def wsattn_plan_ex(frames, tokens_per_frame, window, ref_frames, heads, head_dim, block_q,
                   block_k, mask_flags) -> Plan:
    return wsattn_plan(frames, tokens_per_frame, window, ref_frames, heads, head_dim, block_q,
                       block_k, mask_flags)


def wsattn_plan_destroy(plan: Plan):
    plan.destroy()


def wsattn_prepare(plan: Plan, q, k, stream=None):
    """Key mean, row bounds, row fixed max and per-head eligibility (q, k read only)."""
    import torch
    _check_shape(plan, q, "q")
    _check_shape(plan, k, "k")
    if q.shape[0] != k.shape[0]:
        raise ValueError("q and k batch differ")
    _check(_lib.wsattn_prepare(plan.handle, q.shape[0], _dev_ptr(q, "q", torch.bfloat16),
                               _dev_ptr(k, "k", torch.bfloat16), _stream_ptr(stream)),
           "wsattn_prepare")


def wsattn_produce(plan: Plan, x, w_qkv, rope_cos, rope_sin, eps: float = 1e-6, q=None, k=None,
                   v=None, stream=None):
    """Pre-attention producer: x [B, N, C] bf16, w_qkv [3HD, C] bf16, rope
    tables fp32 [N, D/2] -> (q, k, v) bf16 [B, H, N, D]; the plan's
    statistics are then ready for wsattn_forward, as after wsattn_prepare."""
    import torch
    if x.dim() != 3 or x.shape[1] != plan.n_tokens:
        raise ValueError(f"x must be [B, {plan.n_tokens}, C], got {tuple(x.shape)}")
    B, _, C = x.shape
    hd = plan.heads * plan.head_dim
    if tuple(w_qkv.shape) != (3 * hd, C):
        raise ValueError(f"w_qkv must be [{3 * hd}, {C}], got {tuple(w_qkv.shape)}")
    for t, n in ((rope_cos, "rope_cos"), (rope_sin, "rope_sin")):
        if tuple(t.shape) != (plan.n_tokens, plan.head_dim // 2):
            raise ValueError(f"{n} must be [{plan.n_tokens}, {plan.head_dim // 2}]")
    shape = (B, plan.heads, plan.n_tokens, plan.head_dim)
    q = torch.empty(shape, dtype=torch.bfloat16, device=x.device) if q is None else q
    k = torch.empty(shape, dtype=torch.bfloat16, device=x.device) if k is None else k
    v = torch.empty(shape, dtype=torch.bfloat16, device=x.device) if v is None else v
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check_shape(plan, t, n)
        if t.shape[0] != B:
            raise ValueError(f"{n} batch differs from x")
    _check(_lib.wsattn_produce(plan.handle, B, _dev_ptr(x, "x", torch.bfloat16), C,
                               _dev_ptr(w_qkv, "w_qkv", torch.bfloat16),
                               _dev_ptr(rope_cos, "rope_cos", torch.float32),
                               _dev_ptr(rope_sin, "rope_sin", torch.float32), float(eps),
                               _dev_ptr(q, "q", torch.bfloat16), _dev_ptr(k, "k", torch.bfloat16),
                               _dev_ptr(v, "v", torch.bfloat16), _stream_ptr(stream)),
           "wsattn_produce")
    return q, k, v


def wsattn_forward(plan: Plan, q, k, v, out=None, stream=None):
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check_shape(plan, t, n)
    if not (q.shape[0] == k.shape[0] == v.shape[0]):
        raise ValueError("q, k, v batch differ")
    if out is None:
        out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    _check_shape(plan, out, "out")
    _check(_lib.wsattn_forward(plan.handle, q.shape[0], _dev_ptr(q, "q", torch.bfloat16),
                               _dev_ptr(k, "k", torch.bfloat16), _dev_ptr(v, "v", torch.bfloat16),
                               _dev_ptr(out, "out", torch.float32), _stream_ptr(stream)),
           "wsattn_forward")
    return out


def wsattn_plan_info(plan: Plan) -> dict:
    return {"n_tokens": plan.n_tokens, "block_q": plan.block_q, "block_k": plan.block_k,
            "n_qblocks": plan.n_qblocks, "n_kblocks": plan.n_kblocks, "nnz": plan.nnz,
            "tiles_per_head": plan.tiles_per_head, "head_dim": plan.head_dim,
            "heads": plan.heads, "active_pairs": plan.active_pairs}


def wsattn_get_block_map(plan: Plan) -> np.ndarray:
    out = np.zeros((plan.n_qblocks, plan.n_kblocks), dtype=np.uint8)
    _check(_lib.wsattn_get_block_map(plan.handle, out.ctypes.data, out.size),
           "wsattn_get_block_map")
    return out


def wsattn_get_tiles(plan: Plan):
    """The forward work list: int32 [tiles, 10] {row0, nvalid, nblk, run0, len0,
    run1, nstep, kbeg, gsz, gtab} and the merged tails' group table int32
    [groups, 4] {run0, len0, run1, len1}."""
    tiles = np.zeros((plan.tiles_per_head, 10), dtype=np.int32)
    # each merged tile holds at most 8 row groups (tails of at least 16 rows)
    groups = np.zeros((8 * plan.tiles_per_head, 4), dtype=np.int32)
    _check(_lib.wsattn_get_tiles(plan.handle, tiles.ctypes.data, tiles.size, groups.ctypes.data,
                                 groups.size), "wsattn_get_tiles")
    merged = tiles[:, 8] > 0
    n_groups = int((tiles[merged, 1] // tiles[merged, 8]).sum())  # nvalid = groups x gsz
    return tiles, groups[:n_groups]


def wsattn_get_csr(plan: Plan):
    row_ptr = np.zeros(plan.n_qblocks + 1, dtype=np.int32)
    col = np.zeros(max(plan.nnz, 1), dtype=np.int32)
    _check(_lib.wsattn_get_csr(plan.handle, row_ptr.ctypes.data, col.ctypes.data, row_ptr.size,
                               col.size), "wsattn_get_csr")
    return row_ptr, col[:plan.nnz]


def wsattn_get_stats(plan: Plan, batch: int, stream=None) -> dict:
    bh = batch * plan.heads
    b = np.zeros((bh, plan.n_tokens), dtype=np.float32)
    m = np.zeros((bh, plan.n_tokens), dtype=np.float32)
    mu = np.zeros((bh, plan.head_dim), dtype=np.float32)
    kmax = np.zeros(bh, dtype=np.float32)
    bmax = np.zeros(bh, dtype=np.float32)
    elig = np.zeros(bh, dtype=np.uint8)
    _check(_lib.wsattn_get_stats(plan.handle, b.ctypes.data, m.ctypes.data, mu.ctypes.data,
                                 kmax.ctypes.data, bmax.ctypes.data, elig.ctypes.data,
                                 _stream_ptr(stream)), "wsattn_get_stats")
    return {"b": b, "m": m, "mu": mu, "kmax": kmax, "bmax": bmax, "elig": elig}


def wsattn_plan_set_debug(plan: Plan, force_path: int = -1, tau: float = 0.0):
    _check(_lib.wsattn_plan_set_debug(plan.handle, int(force_path), float(tau)),
           "wsattn_plan_set_debug")


def wsattn_plan_set_bound(plan: Plan, mode: int):
    """BOUND_GLOBAL (default) or BOUND_WINDOW: the key-norm maximum of the row
    bounds; prepare again before the next forward."""
    _check(_lib.wsattn_plan_set_bound(plan.handle, int(mode)), "wsattn_plan_set_bound")


def wsattn_device_status(plan: Plan, stream=None) -> int:
    return int(_lib.wsattn_device_status(plan.handle, _stream_ptr(stream)))


def wsattn_selftest_timeout(limit_ms: int = 50, stream=None) -> int:
    st = _I(-1)
    _check(_lib.wsattn_selftest_timeout(int(limit_ms), ctypes.byref(st), _stream_ptr(stream)),
           "wsattn_selftest_timeout")
    return int(st.value)


def wsattn_prepare_static(q, k, out: dict, tau: float = 40.0, stream=None):
    """No-allocation prepare: statistics into the caller's tensors in `out`
    (keys b, m, mu, kmax, bmax, elig, shaped as wsattn_prepare_static_outputs
    makes them).  For callers that must not let the library allocate."""
    import torch
    B, H, N, D = q.shape
    if k.shape != q.shape:
        raise ValueError("q and k shapes differ")
    _check(_lib.wsattn_prepare_static(
        B, H, N, D, float(tau), _dev_ptr(q, "q", torch.bfloat16), _dev_ptr(k, "k", torch.bfloat16),
        _dev_ptr(out["b"], "b", torch.float32), _dev_ptr(out["m"], "m", torch.float32),
        _dev_ptr(out["mu"], "mu", torch.float32), _dev_ptr(out["kmax"], "kmax", torch.float32),
        _dev_ptr(out["bmax"], "bmax", torch.float32), _dev_ptr(out["elig"], "elig", torch.uint8),
        _stream_ptr(stream)), "wsattn_prepare_static")
    return out


def wsattn_prepare_static_outputs(batch, heads, n_tokens, head_dim, device="cuda"):
    """Caller-owned output tensors for wsattn_prepare_static."""
    import torch
    bh = batch * heads
    f = dict(dtype=torch.float32, device=device)
    return {"b": torch.empty(bh, n_tokens, **f), "m": torch.empty(bh, n_tokens, **f),
            "mu": torch.empty(bh, head_dim, **f), "kmax": torch.empty(bh, **f),
            "bmax": torch.empty(bh, **f),
            "elig": torch.empty(bh, dtype=torch.uint8, device=device)}


def raw_call(name: str):
    """The ctypes function for an exported symbol (for tests of the ABI)."""
    return getattr(_lib, name)
