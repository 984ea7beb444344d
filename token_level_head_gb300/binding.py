"""ctypes binding of the C ABI in ``include/mhla.h`` — argument marshalling only.

Every function here has the name of the C entry point it calls, takes torch
CUDA tensors, passes their device pointers, sizes and the current CUDA stream
to the library, and raises :class:`MhlaError` on a non-OK status.  All work
runs in the library's CUDA kernels; there is no fallback: if the library is
missing or CUDA is unavailable the call fails.
"""

from __future__ import annotations

import ctypes
import os

import torch

from .build import LIB_PATH

MHLA_OK, MHLA_ERR_INVALID_ARG, MHLA_ERR_UNSUPPORTED, MHLA_ERR_CUDA, MHLA_ERR_TIMEOUT = range(5)
MHLA_F32, MHLA_BF16 = 0, 1
PATH_NAMES = {0: "none", 1: "simt", 2: "tcgen05", 3: "tcgen05_stream"}

_lib = None

_vp, _sz, _i, _f = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_float

_SIGNATURES = {
    "mhla_workspace_bytes": (_sz, [_i, _i, _i, _i, _i, _i]),
    "mhla_forward": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _f, _vp, _sz, _vp]),
    "mhla_forward_causal": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _vp, _sz, _vp]),
    "linattn_decode_step": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _vp]),
    "linattn_decode_steps": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _f, _vp]),
    "mhla_causal_stream": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _f, _vp]),
    "mhla_forward_ex": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _f, _vp, _vp, _sz, _vp]),
    "mhla_forward_ex_path": (_i, [_i, _i, _i, _i, _i, _i, _i, _i, _vp]),
    "mhla_forward_grid": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _f, _vp, _sz, _vp]),
    "mhla_forward_grid_path": (_i, [_i, _i, _i, _i, _i, _i, _i, _i]),
    "mhla_locality_mixing": (_i, [_vp, _i, _i]),
    "rala_workspace_bytes": (_sz, [_i, _i, _i, _i, _i]),
    "rala_forward": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp, _sz, _vp]),
    "mhla_forward_path": (_i, [_i, _i, _i, _i, _i, _i, _i]),
    "rala_forward_path": (_i, [_i, _i, _i, _i, _i, _i]),
    "mhla_query_status": (_i, [_vp, _vp]),
    "mhla_status_string": (ctypes.c_char_p, [_i]),
    "mhla_launch_count": (ctypes.c_ulonglong, []),
    "mhla_forward_noalloc": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _vp]),
    "mhla_debug_set_wait_limit_ns": (None, [ctypes.c_ulonglong]),
    "mhla_backward_workspace_bytes": (_sz, [_i, _i, _i, _i, _i]),
    "mhla_backward_path": (_i, [_i, _i, _i, _i, _i, _i]),
    "mhla_backward": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _vp, _sz, _vp]),
}

EXPORTED = tuple(_SIGNATURES)


class MhlaError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {status_string(status)} (status {status})")


def load(path: str = LIB_PATH):
    """Loads the library (once).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(f"MHLA CUDA library not built at {path}; call __graft_entry__.build()")
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype, fn.argtypes = res, args
        _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().mhla_status_string(int(status)).decode()


def _check(fn: str, status: int):
    if status != MHLA_OK:
        raise MhlaError(fn, status)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return MHLA_F32
    if t.dtype == torch.bfloat16:
        return MHLA_BF16
    raise TypeError(f"unsupported dtype {t.dtype}; use float32 or bfloat16")


def _stream(stream, device=None):
    s = torch.cuda.current_stream(device) if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


def _expect(t, name, shape, dtype):
    """Raises ValueError unless tensor ``t`` has this shape and dtype (checked before any device use)."""
    if t is None:
        return
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.dtype != dtype:
        raise ValueError(f"{name}: dtype {t.dtype}, expected {dtype}")


def _same_device(q, *ts):
    """All tensors contiguous on q's CUDA device; returns that device."""
    _need_cuda(q, *ts)
    for t in ts:
        if t is not None and t.device != q.device:
            raise ValueError(f"tensor on {t.device}, expected {q.device} (the device of q)")
    return q.device


def _mhla_args(q, k, v, mixing, y, den_out, block, mixing_required=True):
    if q.dim() != 4:
        raise ValueError(f"q: expected [B, H, N, d], got shape {tuple(q.shape)}")
    B, H, N, d = q.shape
    for name, t in (("k", k), ("v", v), ("y", y)):
        _expect(t, name, q.shape, q.dtype)
    _expect(den_out, "den_out", (B, H, N), torch.float32)
    if mixing is None:
        if mixing_required:
            raise ValueError("mixing: required")
    elif block > 0 and N % block == 0:
        _expect(mixing, "mixing", (H, N // block, N // block), torch.float32)
    return B, H, N, d


def mhla_workspace_bytes(B: int, H: int, N: int, d: int, block_size: int, causal: int = 0) -> int:
    return int(load().mhla_workspace_bytes(B, H, N, d, block_size, causal))


def mhla_backward_workspace_bytes(B: int, H: int, N: int, d: int, block_size: int) -> int:
    return int(load().mhla_backward_workspace_bytes(B, H, N, d, block_size))


def rala_workspace_bytes(B: int, H: int, N: int, d: int, cx: int) -> int:
    return int(load().rala_workspace_bytes(B, H, N, d, cx))


def new_workspace(nbytes: int, device) -> torch.Tensor:
    """Zero-filled uint8 device buffer of ``nbytes`` (the library needs it zeroed before first use)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def mhla_forward_path(B, H, N, d, block_size, causal, dtype) -> str:
    dt = MHLA_BF16 if dtype == torch.bfloat16 else MHLA_F32
    return PATH_NAMES[int(load().mhla_forward_path(B, H, N, d, block_size, causal, dt))]


def mhla_forward_grid_path(B, H, grid_h, grid_w, tile_h, tile_w, d, dtype) -> str:
    dt = MHLA_BF16 if dtype == torch.bfloat16 else MHLA_F32
    return PATH_NAMES[int(load().mhla_forward_grid_path(B, H, grid_h, grid_w, tile_h, tile_w, d, dt))]


def locality_mixing(blocks_h, blocks_w) -> torch.Tensor:
    """The locality-based initial mixing matrix [M, M] (fp32, CPU) for blocks on a grid."""
    M = blocks_h * blocks_w
    m = torch.empty(max(M, 0), max(M, 0), dtype=torch.float32)
    _check("mhla_locality_mixing", load().mhla_locality_mixing(_ptr(m), blocks_h, blocks_w))
    return m


def rala_forward_path(B, H, N, d, cx, dtype) -> str:
    dt = MHLA_BF16 if dtype == torch.bfloat16 else MHLA_F32
    return PATH_NAMES[int(load().rala_forward_path(B, H, N, d, cx, dt))]


# Every wrapper checks shapes and dtypes against q, then that every tensor is a
# contiguous CUDA tensor on q's device, and runs the call with q's device
# current (the library takes its device from the current device).

def mhla_forward(q, k, v, mixing, y, block_size, *, causal=0, eps=1e-6, den_out=None,
                 workspace=None, stream=None):
    """Non-causal (or, with causal=1, causal) MHLA forward; q/k/v/y [B, H, N, d], mixing [H, M, M] fp32."""
    B, H, N, d = _mhla_args(q, k, v, mixing, y, den_out, block_size, mixing_required=not causal)
    dev = _same_device(q, k, v, mixing, y, den_out, workspace)
    with torch.cuda.device(dev):
        if workspace is None:
            workspace = new_workspace(mhla_workspace_bytes(B, H, N, d, block_size, causal), dev)
        st = load().mhla_forward(_ptr(q), _ptr(k), _ptr(v), _ptr(mixing), _ptr(y), _ptr(den_out),
                                 B, H, N, d, block_size, causal, _dtype(q), eps, _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), _stream(stream, dev))
    _check("mhla_forward", st)
    return y


FEATURES = {"elu1": 0, "relu": 1, "exp": 2}


class MhlaOptions(ctypes.Structure):
    """The C struct mhla_options: feature map, normaliser on / off, causal decay."""
    _fields_ = [("feature", ctypes.c_int), ("normalise", ctypes.c_int), ("gamma", ctypes.c_float)]


def _options(feature, normalise, gamma):
    if feature not in FEATURES:
        raise ValueError(f"feature: one of {sorted(FEATURES)}, got {feature!r}")
    return MhlaOptions(FEATURES[feature], 1 if normalise else 0, float(gamma))


def mhla_forward_ex_path(B, H, N, d, block_size, causal, with_mixing, dtype, *, feature="elu1", normalise=True,
                         gamma=1.0) -> str:
    dt = MHLA_BF16 if dtype == torch.bfloat16 else MHLA_F32
    opt = _options(feature, normalise, gamma)
    return PATH_NAMES[int(load().mhla_forward_ex_path(B, H, N, d, block_size, causal, int(bool(with_mixing)), dt,
                                                      ctypes.byref(opt)))]


def mhla_forward_ex(q, k, v, mixing, y, block_size, *, causal=0, feature="elu1", normalise=True, gamma=1.0,
                    eps=1e-6, den_out=None, workspace=None, stream=None):
    """mhla_forward with variants: feature map ("elu1", "relu", "exp"), normalise (False: the
    numerator alone), gamma (decay; plain causal linear attention, mixing None, only)."""
    opt = _options(feature, normalise, gamma)
    B, H, N, d = _mhla_args(q, k, v, mixing, y, den_out, block_size, mixing_required=not causal)
    dev = _same_device(q, k, v, mixing, y, den_out, workspace)
    with torch.cuda.device(dev):
        if workspace is None:
            workspace = new_workspace(mhla_workspace_bytes(B, H, N, d, block_size, causal), dev)
        st = load().mhla_forward_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(mixing), _ptr(y), _ptr(den_out),
                                    B, H, N, d, block_size, causal, _dtype(q), eps, ctypes.byref(opt),
                                    _ptr(workspace), workspace.numel() * workspace.element_size(),
                                    _stream(stream, dev))
    _check("mhla_forward_ex", st)
    return y


def mhla_forward_grid(q, k, v, mixing, y, grid_hw, tile_hw, *, eps=1e-6, den_out=None, workspace=None,
                      stream=None):
    """Non-causal MHLA with 2-D blocks: the N tokens are a grid_hw = (grid_h, grid_w) grid in
    row-major order, the blocks its tile_hw = (tile_h, tile_w) tiles; mixing [H, M, M] fp32."""
    (gh, gw), (th, tw) = grid_hw, tile_hw
    if q.dim() != 4:
        raise ValueError(f"q: expected [B, H, N, d], got shape {tuple(q.shape)}")
    if q.shape[2] != gh * gw:
        raise ValueError(f"q: N = {q.shape[2]}, expected grid_h * grid_w = {gh * gw}")
    if th <= 0 or tw <= 0 or gh % th or gw % tw:
        raise ValueError(f"tiles {tile_hw} do not cover the grid {grid_hw}")
    B, H, N, d = q.shape
    for name, t in (("k", k), ("v", v), ("y", y)):
        _expect(t, name, q.shape, q.dtype)
    _expect(den_out, "den_out", (B, H, N), torch.float32)
    M = (gh // th) * (gw // tw)
    _expect(mixing, "mixing", (H, M, M), torch.float32)
    dev = _same_device(q, k, v, mixing, y, den_out, workspace)
    with torch.cuda.device(dev):
        if workspace is None:
            workspace = new_workspace(mhla_workspace_bytes(B, H, N, d, th * tw, 0), dev)
        st = load().mhla_forward_grid(_ptr(q), _ptr(k), _ptr(v), _ptr(mixing), _ptr(y), _ptr(den_out),
                                      B, H, gh, gw, th, tw, d, _dtype(q), eps, _ptr(workspace),
                                      workspace.numel() * workspace.element_size(), _stream(stream, dev))
    _check("mhla_forward_grid", st)
    return y


def mhla_causal_stream(q, k, v, mixing, S, z, out, t0, block, *, eps=1e-6, den_out=None, stream=None):
    """Causal MHLA inference for tokens t0 .. t0 + T - 1: q/k/v/out [T, B, H, d], mixing [H, M, M]
    fp32, S [B, H, M, d, d] and z [B, H, M, d] fp32 block summaries (updated)."""
    if q.dim() != 4 or S.dim() != 5:
        raise ValueError("q: expected [T, B, H, d]; S: expected [B, H, M, d, d]")
    T, B, H, d = q.shape
    M = S.shape[2]
    for name, t in (("k", k), ("v", v), ("out", out)):
        _expect(t, name, q.shape, q.dtype)
    _expect(mixing, "mixing", (H, M, M), torch.float32)
    _expect(S, "S", (B, H, M, d, d), torch.float32)
    _expect(z, "z", (B, H, M, d), torch.float32)
    _expect(den_out, "den_out", (T, B, H), torch.float32)
    dev = _same_device(q, k, v, mixing, S, z, out, den_out)
    with torch.cuda.device(dev):
        st = load().mhla_causal_stream(_ptr(q), _ptr(k), _ptr(v), _ptr(mixing), _ptr(S), _ptr(z), _ptr(out),
                                       _ptr(den_out), t0, T, B, H, d, block, M, _dtype(q), eps,
                                       _stream(stream, dev))
    _check("mhla_causal_stream", st)
    return out


def mhla_forward_causal(q, k, v, mixing, y, chunk, *, eps=1e-6, den_out=None, workspace=None,
                        stream=None):
    """Causal chunked forward; mixing None = plain causal linear attention."""
    B, H, N, d = _mhla_args(q, k, v, mixing, y, den_out, chunk, mixing_required=False)
    dev = _same_device(q, k, v, mixing, y, den_out, workspace)
    with torch.cuda.device(dev):
        if workspace is None:
            workspace = new_workspace(mhla_workspace_bytes(B, H, N, d, chunk, 1), dev)
        st = load().mhla_forward_causal(_ptr(q), _ptr(k), _ptr(v), _ptr(mixing), _ptr(y), _ptr(den_out),
                                        B, H, N, d, chunk, _dtype(q), eps, _ptr(workspace),
                                        workspace.numel() * workspace.element_size(), _stream(stream, dev))
    _check("mhla_forward_causal", st)
    return y


def mhla_backward_path(B, H, N, d, block_size, dtype) -> str:
    dt = MHLA_BF16 if dtype == torch.bfloat16 else MHLA_F32
    return PATH_NAMES[int(load().mhla_backward_path(B, H, N, d, block_size, dt))]


def mhla_backward(q, k, v, mixing, dy, dq, dk, dv, dmixing, block_size, *, eps=1e-6, workspace=None, stream=None):
    """Gradients of the non-causal MHLA forward: dq, dk, dv [B, H, N, d] (q's dtype) and dmixing
    [H, M, M] fp32 from dy = dL/dY; all four are written."""
    B, H, N, d = _mhla_args(q, k, v, mixing, dy, None, block_size)
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        _expect(t, name, q.shape, q.dtype)
    _expect(dmixing, "dmixing", mixing.shape, torch.float32)
    dev = _same_device(q, k, v, mixing, dy, dq, dk, dv, dmixing, workspace)
    with torch.cuda.device(dev):
        if workspace is None:
            workspace = new_workspace(mhla_backward_workspace_bytes(B, H, N, d, block_size), dev)
        st = load().mhla_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(mixing), _ptr(dy), _ptr(dq), _ptr(dk), _ptr(dv),
                                  _ptr(dmixing), B, H, N, d, block_size, _dtype(q), eps, _ptr(workspace),
                                  workspace.numel() * workspace.element_size(), _stream(stream, dev))
    _check("mhla_backward", st)
    return dq, dk, dv, dmixing


def linattn_decode_step(q, k, v, S, z, out, *, eps=1e-6, den_out=None, stream=None):
    """One recurrent decode step; q/k/v/out [B, H, d], S [B, H, d, d] fp32, z [B, H, d] fp32 (updated)."""
    if q.dim() != 3:
        raise ValueError(f"q: expected [B, H, d], got shape {tuple(q.shape)}")
    B, H, d = q.shape
    for name, t in (("k", k), ("v", v), ("out", out)):
        _expect(t, name, q.shape, q.dtype)
    _expect(S, "S", (B, H, d, d), torch.float32)
    _expect(z, "z", (B, H, d), torch.float32)
    _expect(den_out, "den_out", (B, H), torch.float32)
    dev = _same_device(q, k, v, S, z, out, den_out)
    with torch.cuda.device(dev):
        st = load().linattn_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(S), _ptr(z), _ptr(out),
                                        _ptr(den_out), B, H, d, _dtype(q), eps, _stream(stream, dev))
    _check("linattn_decode_step", st)
    return out


def linattn_decode_steps(q, k, v, S, z, out, *, eps=1e-6, gamma=1.0, den_out=None, stream=None):
    """T recurrent decode steps in one call; q/k/v/out [T, B, H, d], S [B, H, d, d] fp32,
    z [B, H, d] fp32 (updated), den_out [T, B, H] fp32; ``gamma`` the decay in [0, 1]."""
    if q.dim() != 4:
        raise ValueError(f"q: expected [T, B, H, d], got shape {tuple(q.shape)}")
    T, B, H, d = q.shape
    for name, t in (("k", k), ("v", v), ("out", out)):
        _expect(t, name, q.shape, q.dtype)
    _expect(S, "S", (B, H, d, d), torch.float32)
    _expect(z, "z", (B, H, d), torch.float32)
    _expect(den_out, "den_out", (T, B, H), torch.float32)
    dev = _same_device(q, k, v, S, z, out, den_out)
    with torch.cuda.device(dev):
        st = load().linattn_decode_steps(_ptr(q), _ptr(k), _ptr(v), _ptr(S), _ptr(z), _ptr(out),
                                         _ptr(den_out), T, B, H, d, _dtype(q), eps, gamma,
                                         _stream(stream, dev))
    _check("linattn_decode_steps", st)
    return out


def rala_forward(q, k, v, x, w, y, *, workspace=None, stream=None):
    """Rank-augmented linear attention; q/k/v/y [B, H, N, d], x [B, N, cx], w [cx, d]."""
    if q.dim() != 4 or x.dim() != 3:
        raise ValueError("q: expected [B, H, N, d]; x: expected [B, N, cx]")
    B, H, N, d = q.shape
    cx = x.shape[-1]
    for name, t in (("k", k), ("v", v), ("y", y)):
        _expect(t, name, q.shape, q.dtype)
    _expect(x, "x", (B, N, cx), q.dtype)
    _expect(w, "w", (cx, d), q.dtype)
    dev = _same_device(q, k, v, x, w, y, workspace)
    with torch.cuda.device(dev):
        if workspace is None:
            workspace = new_workspace(rala_workspace_bytes(B, H, N, d, cx), dev)
        st = load().rala_forward(_ptr(q), _ptr(k), _ptr(v), _ptr(x), _ptr(w), _ptr(y), B, H, N, d, cx,
                                 _dtype(q), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                 _stream(stream, dev))
    _check("rala_forward", st)
    return y


def mhla_forward_noalloc(q, k, v, mixing, y, block_size, *, eps=1e-6, den_out=None, stream=None):
    """Non-causal MHLA forward with no workspace: for callers that cannot allocate device memory.

    The library keeps a fixed 32 MiB scratch array per GPU for it; calls that
    overlap on the GPU share that array and must not run concurrently.
    """
    B, H, N, d = _mhla_args(q, k, v, mixing, y, den_out, block_size)
    dev = _same_device(q, k, v, mixing, y, den_out)
    with torch.cuda.device(dev):
        st = load().mhla_forward_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(mixing), _ptr(y), _ptr(den_out),
                                         B, H, N, d, block_size, _dtype(q), eps, _stream(stream, dev))
    _check("mhla_forward_noalloc", st)
    return y


def mhla_query_status(workspace, stream=None) -> int:
    with torch.cuda.device(workspace.device):
        return int(load().mhla_query_status(_ptr(workspace), _stream(stream, workspace.device)))


def mhla_launch_count() -> int:
    return int(load().mhla_launch_count())


def mhla_debug_set_wait_limit_ns(ns: int) -> None:
    """Diagnostic: limit of the device-side waits of the bf16 tensor-core forward (0 = default)."""
    load().mhla_debug_set_wait_limit_ns(int(ns))
