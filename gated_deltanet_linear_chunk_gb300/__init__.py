"""GB300 (sm_103a) Gated DeltaNet layer: chunked prefill and recurrent decode.

The compute lives in ``libgdn`` (hand-written CUDA behind the C ABI declared
in ``include/gdn.h``).  This module is the thin binding: it checks tensor
shapes and dtypes, marshals device pointers and the current CUDA stream, and
calls the C entry points of the same names.  Every step of the layer runs in
the library's kernels; there is no other implementation to fall back on, and
a missing library raises.

Method: per token ``S_t = a_t S_{t-1} (I - b_t k_t k_t^T) + b_t v_t k_t^T``,
``o_t = S_t q_t`` with ``a_t = exp(g_t)`` (Gated DeltaNet, the linear-attention
layers of the hybrid Qwen3.8-27B model; page "cf-1.com", section "三个优化",
item 2 "GDN prefill", chunk length 64).
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

import torch

from . import build as _build

__all__ = [
    "GDNError", "library", "gdn_chunk_prefill", "gdn_decode_step",
    "gdn_chunk_prefill_workspace_size", "gdn_chunk_prefill_noalloc", "gdn_status_string",
    "gdn_version", "gdn_chunk_prefill_device_status", "gdn_decode_step_half_state",
    "gdn_verify_step", "gdn_chunk_prefill_snapshots", "gdn_chunk_prefill_snapshot_slots",
    "gdn_chunk_prefill_timed", "gdn_prefill_fused_mode", "gdn_prefill_path",
    "gdn_chunk_prefill_host",
    "gdn_chunk_prefill_scan",
    "gdn_chunk_prefill_scan_workspace_size", "Problem",
    "GDN_BF16", "GDN_F32",
]

GDN_BF16 = 0
GDN_F32 = 1
GDN_F16 = 2  # state storage of gdn_decode_step_half_state only

# gdn_status codes (include/gdn.h).
GDN_OK = 0
GDN_ERR_INVALID_ARG = 1
GDN_ERR_UNSUPPORTED = 2
GDN_ERR_MISALIGNED = 3
GDN_ERR_WORKSPACE = 4
GDN_ERR_CUDA = 5
GDN_ERR_TIMEOUT = 6
GDN_ERR_INTERNAL = 7  # a device-side index check of a GDN_DEBUG build failed
_DTYPES = {torch.bfloat16: GDN_BF16, torch.float32: GDN_F32}


class Problem(ctypes.Structure):
    """Mirror of ``gdn_problem`` in include/gdn.h."""

    _fields_ = [
        ("num_seqs", ctypes.c_int32),
        ("total_tokens", ctypes.c_int64),
        ("num_k_heads", ctypes.c_int32),
        ("num_v_heads", ctypes.c_int32),
        ("head_dim_k", ctypes.c_int32),
        ("head_dim_v", ctypes.c_int32),
        ("qkv_dtype", ctypes.c_int32),
        ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t),
    ]


class GDNError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = int(code)
        super().__init__(f"{where}: {gdn_status_string(code)}")


_lib = None


def library() -> ctypes.CDLL:
    """The loaded CUDA library; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    _lib = _load(_build.library_path())
    return _lib


_debug_lib = None


def debug_library() -> ctypes.CDLL:
    """The GDN_DEBUG variant of the library (the same C ABI; the kernels also
    check the inputs' preconditions and their own indices on the device and
    report through gdn_chunk_prefill_device_status).  The wrappers of this
    module call library(); this one is called through its C ABI directly."""
    global _debug_lib
    if _debug_lib is None:
        _debug_lib = _load(_build.library_path(debug=True))
    return _debug_lib


def _load(path: str) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise RuntimeError(
            f"the CUDA library {path} is missing: build it first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    PP = ctypes.POINTER(Problem)
    lib.gdn_chunk_prefill_workspace_size.restype = ctypes.c_size_t
    lib.gdn_chunk_prefill_workspace_size.argtypes = [PP]
    lib.gdn_chunk_prefill.restype = ctypes.c_int
    lib.gdn_chunk_prefill.argtypes = [PP, P, P, P, P, P, P, P, P, P, P]
    lib.gdn_chunk_prefill_noalloc.restype = ctypes.c_int
    lib.gdn_chunk_prefill_noalloc.argtypes = [PP, P, P, P, P, P, P, P, P, P, P]
    lib.gdn_decode_step.restype = ctypes.c_int
    lib.gdn_decode_step.argtypes = [PP, P, P, P, P, P, P, P, P]
    lib.gdn_status_string.restype = ctypes.c_char_p
    lib.gdn_status_string.argtypes = [ctypes.c_int]
    lib.gdn_version.restype = ctypes.c_int
    lib.gdn_version.argtypes = []
    lib.gdn_decode_step_half_state.restype = ctypes.c_int
    lib.gdn_decode_step_half_state.argtypes = [PP, P, P, P, P, P, P, ctypes.c_int32, P, P]
    lib.gdn_chunk_prefill_snapshot_slots.restype = ctypes.c_int64
    lib.gdn_chunk_prefill_snapshot_slots.argtypes = [PP, ctypes.c_int32]
    lib.gdn_chunk_prefill_snapshots.restype = ctypes.c_int
    lib.gdn_chunk_prefill_snapshots.argtypes = [PP, P, P, P, P, P, P, P, P, P, P, ctypes.c_int32,
                                                P]
    lib.gdn_verify_step.restype = ctypes.c_int
    lib.gdn_verify_step.argtypes = [PP, ctypes.c_int32, P, P, P, P, P, P, ctypes.c_int32, P, P, P]
    lib.gdn_chunk_prefill_device_status.restype = ctypes.c_int
    lib.gdn_chunk_prefill_device_status.argtypes = [P, P]
    lib.gdn_chunk_prefill_scan_workspace_size.restype = ctypes.c_size_t
    lib.gdn_chunk_prefill_scan_workspace_size.argtypes = [PP, ctypes.c_int32]
    lib.gdn_chunk_prefill_scan.restype = ctypes.c_int
    lib.gdn_chunk_prefill_scan.argtypes = [PP, ctypes.c_int32] + [P] * 10
    lib.gdn_chunk_prefill_timed.restype = ctypes.c_int
    lib.gdn_chunk_prefill_timed.argtypes = [PP, P, P, P, P, P, P, P, P, P, P, P, P]
    lib.gdn_chunk_prefill_prep_only.restype = ctypes.c_int
    lib.gdn_chunk_prefill_prep_only.argtypes = [PP, P, P, P, P, P, P]
    lib.gdn_chunk_prefill_prep_layout.restype = ctypes.c_int
    lib.gdn_chunk_prefill_prep_layout.argtypes = [PP, P]
    lib.gdn_chunk_prefill_host.restype = ctypes.c_int
    lib.gdn_chunk_prefill_host.argtypes = [PP, ctypes.c_int32] + [P] * 16 + [P]
    lib.gdn_prefill_fused_mode.restype = ctypes.c_int32
    lib.gdn_prefill_fused_mode.argtypes = [ctypes.c_int32]
    lib.gdn_prefill_path.restype = ctypes.c_int32
    lib.gdn_prefill_path.argtypes = [PP, ctypes.c_int32, ctypes.c_int32]
    return lib


_staging = threading.local()  # per host thread: .key, .bufs


def gdn_chunk_prefill_host(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                           g: torch.Tensor, beta: torch.Tensor, out: torch.Tensor,
                           initial_state: Optional[torch.Tensor] = None,
                           final_state: Optional[torch.Tensor] = None, pieces: int = 4,
                           device=None, stream=None) -> torch.Tensor:
    """Prefill of one sequence whose q, k, v, g, beta and out live in (pinned)
    host memory; the transfers overlap the computation (see
    ``gdn_chunk_prefill_host`` in include/gdn.h).  initial_state and
    final_state, if given, are device tensors [1, Hv, dv, dk].  The device
    staging buffers are kept per host thread for the last shape, so calls
    from several threads do not share them.  Returns out."""
    T, Hk, dk = q.shape
    Hv, dv = v.shape[1], v.shape[2]
    dt = q.dtype
    if dt not in _DTYPES:
        raise TypeError(f"unsupported q/k/v dtype {dt}")
    for t, name, tdt, shape in ((q, "q", dt, (T, Hk, dk)), (k, "k", dt, (T, Hk, dk)),
                                (v, "v", dt, (T, Hv, dv)), (g, "g", torch.float32, (T, Hv)),
                                (beta, "beta", torch.float32, (T, Hv)),
                                (out, "out", dt, (T, Hv, dv))):
        if t.device.type != "cpu" or t.dtype != tdt or tuple(t.shape) != shape or \
                not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous host tensor {tdt} {shape}")
    dev = torch.device(device if device is not None else "cuda")
    if dev.index is None:
        dev = torch.device("cuda", torch.cuda.current_device())
    cs = _stream_obj(stream, dev)
    key = (dev.index, T, Hk, Hv, dk, dv, dt)
    st = getattr(_staging, "bufs", None) if getattr(_staging, "key", None) == key else None
    done = getattr(_staging, "done", None)  # (stream handle, event) of the last call
    if st is None:
        if done is not None:
            done[1].synchronize()  # the old buffers may still be in use
            done = _staging.done = None
        with torch.cuda.stream(cs):
            st = dict(q=torch.empty((T, Hk, dk), dtype=dt, device=dev),
                      k=torch.empty((T, Hk, dk), dtype=dt, device=dev),
                      v=torch.empty((T, Hv, dv), dtype=dt, device=dev),
                      g=torch.empty((T, Hv), dtype=torch.float32, device=dev),
                      beta=torch.empty((T, Hv), dtype=torch.float32, device=dev),
                      out=torch.empty((T, Hv, dv), dtype=dt, device=dev),
                      cu=torch.empty(128, dtype=torch.int32, device=dev),
                      state=torch.empty((Hv, dv, dk), dtype=torch.float32, device=dev))
        _staging.key, _staging.bufs = key, st
    elif done is not None and done[0] != cs.cuda_stream:
        cs.wait_event(done[1])  # the last call on these buffers ran on another stream
    for t, name in ((initial_state, "initial_state"), (final_state, "final_state")):
        if t is not None:
            _check(t, name, torch.float32, (1, Hv, dv, dk))
    _same_device(dev, initial_state=initial_state, final_state=final_state)
    lib = library()
    p = make_problem(1, T, Hk, Hv, dk, dv, dt)
    need = int(lib.gdn_chunk_prefill_workspace_size(ctypes.byref(p)))
    ws = _workspace(dev, need, cs)
    p = make_problem(1, T, Hk, Hv, dk, dv, dt, ws)
    with torch.cuda.device(dev):
        rc = lib.gdn_chunk_prefill_host(
            ctypes.byref(p), int(pieces), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(out),
            _ptr(initial_state), _ptr(final_state), _ptr(st["q"]), _ptr(st["k"]), _ptr(st["v"]),
            _ptr(st["g"]), _ptr(st["beta"]), _ptr(st["out"]), _ptr(st["cu"]), _ptr(st["state"]),
            cs.cuda_stream)
    if rc != 0:
        raise GDNError(rc, "gdn_chunk_prefill_host")
    ev = torch.cuda.Event()
    ev.record(cs)
    _staging.done = (cs.cuda_stream, ev)
    return out


def gdn_prefill_fused_mode(mode: int = -1) -> int:
    """Sets when prefills use the fused prep + recurrence kernel (0 never,
    1 whenever possible, 2 when expected faster, 3 the variant with one
    recurrence per value head whenever possible; default 2) and returns the
    previous mode; -1 only queries."""
    return int(library().gdn_prefill_fused_mode(int(mode)))


def gdn_prefill_path(num_seqs: int, total_tokens: int, Hk: int, Hv: int, dk: int = 128,
                     dv: int = 128, sms: int = 152, mode: int = -1,
                     dtype=torch.bfloat16) -> int:
    """Which kernels a prefill of this size would run on a GPU with `sms` SMs
    (see ``gdn_prefill_path`` in include/gdn.h): 0 separate, 1 fused, 2 fused
    with one recurrence per value head; -1 without the tensor-core path.
    Needs no device."""
    p = make_problem(num_seqs, total_tokens, Hk, Hv, dk, dv, dtype)
    return int(library().gdn_prefill_path(ctypes.byref(p), int(sms), int(mode)))


def gdn_status_string(code: int) -> str:
    return library().gdn_status_string(int(code)).decode()


def gdn_version() -> int:
    return int(library().gdn_version())


def make_problem(num_seqs: int, total_tokens: int, Hk: int, Hv: int, dk: int, dv: int,
                 dtype, workspace: Optional[torch.Tensor] = None) -> Problem:
    code = _DTYPES[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    ws_ptr = None if workspace is None else workspace.data_ptr()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return Problem(num_seqs, total_tokens, Hk, Hv, dk, dv, code, ws_ptr, ws_bytes)


def gdn_chunk_prefill_workspace_size(num_seqs: int, total_tokens: int, Hk: int, Hv: int,
                                     dk: int, dv: int, dtype=torch.bfloat16) -> int:
    p = make_problem(num_seqs, total_tokens, Hk, Hv, dk, dv, dtype)
    return int(library().gdn_chunk_prefill_workspace_size(ctypes.byref(p)))


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _same_device(dev: torch.device, **tensors) -> None:
    """Every given tensor must live on `dev` (the device the call runs on):
    a tensor on another GPU would be read through pointers that mean nothing
    on this one."""
    for name, t in tensors.items():
        if t is not None and t.device != dev:
            raise ValueError(f"{name} is on {t.device}, but q is on {dev}: all tensors of a "
                             "call must be on one device")


def _check(t: torch.Tensor, name: str, dtype, shape) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


# Prefill scratch kept by this module, one per (device, stream, host thread):
# calls that could run concurrently never share one, and each is allocated on
# the stream that uses it, so the caching allocator reuses it only after that
# stream's work.
_workspaces = {}
_NO_SNAPSHOTS = object()


def _stream_obj(stream, device: torch.device):
    """The torch stream object for `stream` (None: the current stream)."""
    if stream is None:
        return torch.cuda.current_stream(device)
    if hasattr(stream, "cuda_stream"):
        return stream
    return torch.cuda.ExternalStream(int(stream), device=device)


def _workspace_key(device: torch.device, stream) -> tuple:
    dev = device.index if device.index is not None else torch.cuda.current_device()
    dev = torch.device("cuda", dev)
    return (dev.index, _stream_obj(stream, dev).cuda_stream, threading.get_ident())


def _workspace(device: torch.device, nbytes: int, stream=None) -> Optional[torch.Tensor]:
    if nbytes == 0:
        return None
    key = _workspace_key(device, stream)
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < nbytes:
        with torch.cuda.stream(_stream_obj(stream, torch.device("cuda", key[0]))):
            ws = torch.empty(nbytes, dtype=torch.uint8, device=torch.device("cuda", key[0]))
        _workspaces[key] = ws
    return ws


def gdn_chunk_prefill_snapshot_slots(N: int, T: int, Hk: int, Hv: int, dk: int, dv: int,
                                     snapshot_chunks: int = 1, dtype=torch.bfloat16) -> int:
    """Slots gdn_chunk_prefill_snapshots needs (0 if unsupported)."""
    p = make_problem(N, T, Hk, Hv, dk, dv, dtype)
    return int(library().gdn_chunk_prefill_snapshot_slots(ctypes.byref(p), snapshot_chunks))


def gdn_chunk_prefill(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                      g: torch.Tensor, beta: torch.Tensor, cu_seqlens: torch.Tensor,
                      initial_state: Optional[torch.Tensor] = None,
                      out: Optional[torch.Tensor] = None,
                      final_state: Optional[torch.Tensor] = None,
                      output_final_state: bool = False,
                      workspace: Optional[torch.Tensor] = None,
                      stream=None) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Chunked GDN prefill over packed sequences (see ``gdn_chunk_prefill`` in
    include/gdn.h).  q, k: [T, Hk, dk]; v: [T, Hv, dv]; g, beta: [T, Hv] fp32;
    cu_seqlens: [N+1] int32 on the device.  Returns (out, final_state); the
    final state is returned when ``final_state`` is given or
    ``output_final_state`` is set."""
    return _prefill(q, k, v, g, beta, cu_seqlens, initial_state, out, final_state,
                    output_final_state, workspace, stream, _NO_SNAPSHOTS, 0)


def _prefill(q, k, v, g, beta, cu_seqlens, initial_state, out, final_state, output_final_state,
             workspace, stream, snapshots, snapshot_chunks, scan_group=None, events=None):
    """Checks, workspace and dispatch of the prefill entry points
    (``snapshots``: _NO_SNAPSHOTS, None to allocate, or a tensor; ``events``:
    four torch.cuda.Event for the timed call).  Every tensor must be on q's
    device; the call runs with that device current."""
    T, Hk, dk = q.shape
    Hv, dv = v.shape[1], v.shape[2]
    N = cu_seqlens.shape[0] - 1
    dt = q.dtype
    if dt not in _DTYPES:
        raise TypeError(f"unsupported q/k/v dtype {dt}")
    _check(q, "q", dt, (T, Hk, dk))
    _check(k, "k", dt, (T, Hk, dk))
    _check(v, "v", dt, (T, Hv, dv))
    _check(g, "g", torch.float32, (T, Hv))
    _check(beta, "beta", torch.float32, (T, Hv))
    _check(cu_seqlens, "cu_seqlens", torch.int32, (N + 1,))
    if initial_state is not None:
        _check(initial_state, "initial_state", torch.float32, (N, Hv, dv, dk))
    if out is None:
        out = torch.empty((T, Hv, dv), dtype=dt, device=q.device)
    _check(out, "out", dt, (T, Hv, dv))
    if final_state is None and output_final_state:
        final_state = torch.empty((N, Hv, dv, dk), dtype=torch.float32, device=q.device)
    if final_state is not None:
        _check(final_state, "final_state", torch.float32, (N, Hv, dv, dk))
    _same_device(q.device, k=k, v=v, g=g, beta=beta, cu_seqlens=cu_seqlens,
                 initial_state=initial_state, out=out, final_state=final_state,
                 workspace=workspace,
                 snapshots=None if snapshots is _NO_SNAPSHOTS else snapshots)
    with torch.cuda.device(q.device):
        lib = library()
        p = make_problem(N, T, Hk, Hv, dk, dv, dt)
        if scan_group is not None:
            need = int(lib.gdn_chunk_prefill_scan_workspace_size(ctypes.byref(p), scan_group))
            if need == 0 and N > 0:
                raise GDNError(GDN_ERR_UNSUPPORTED, "gdn_chunk_prefill_scan")
        else:
            need = int(lib.gdn_chunk_prefill_workspace_size(ctypes.byref(p)))
        if workspace is None:
            workspace = _workspace(q.device, need, stream)
        p = make_problem(N, T, Hk, Hv, dk, dv, dt, workspace)
        if scan_group is not None:
            rc = lib.gdn_chunk_prefill_scan(ctypes.byref(p), scan_group, _ptr(q), _ptr(k),
                                            _ptr(v), _ptr(g), _ptr(beta), _ptr(cu_seqlens),
                                            _ptr(initial_state), _ptr(out), _ptr(final_state),
                                            _stream(stream))
            if rc != 0:
                raise GDNError(rc, "gdn_chunk_prefill_scan")
            return out, final_state
        if events is not None:
            st = _stream_obj(stream, q.device)
            for e in events:
                e.record(st)  # creates the event (torch creates it lazily)
            handles = (ctypes.c_void_p * 4)(*[e.cuda_event for e in events])
            fused = ctypes.c_int32(0)
            rc = lib.gdn_chunk_prefill_timed(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v),
                                             _ptr(g), _ptr(beta), _ptr(cu_seqlens),
                                             _ptr(initial_state), _ptr(out), _ptr(final_state),
                                             ctypes.cast(handles, ctypes.c_void_p),
                                             ctypes.addressof(fused), st.cuda_stream)
            if rc != 0:
                raise GDNError(rc, "gdn_chunk_prefill_timed")
            return out, final_state, int(fused.value)
        if snapshots is _NO_SNAPSHOTS:
            rc = lib.gdn_chunk_prefill(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                       _ptr(beta), _ptr(cu_seqlens), _ptr(initial_state),
                                       _ptr(out), _ptr(final_state), _stream(stream))
            if rc != 0:
                raise GDNError(rc, "gdn_chunk_prefill")
            return out, final_state
        slots = int(lib.gdn_chunk_prefill_snapshot_slots(ctypes.byref(p), snapshot_chunks))
        if slots == 0:
            raise GDNError(GDN_ERR_UNSUPPORTED, "gdn_chunk_prefill_snapshots")
        if snapshots is None:
            snapshots = torch.empty((slots, Hv, dv, dk), dtype=torch.float32, device=q.device)
        _check(snapshots, "snapshots", torch.float32, (slots, Hv, dv, dk))
        rc = lib.gdn_chunk_prefill_snapshots(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v),
                                             _ptr(g), _ptr(beta), _ptr(cu_seqlens),
                                             _ptr(initial_state), _ptr(out), _ptr(final_state),
                                             _ptr(snapshots), snapshot_chunks, _stream(stream))
        if rc != 0:
            raise GDNError(rc, "gdn_chunk_prefill_snapshots")
        return out, final_state, snapshots


def gdn_chunk_prefill_timed(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                            g: torch.Tensor, beta: torch.Tensor, cu_seqlens: torch.Tensor,
                            initial_state: Optional[torch.Tensor] = None,
                            out: Optional[torch.Tensor] = None,
                            final_state: Optional[torch.Tensor] = None,
                            output_final_state: bool = False,
                            events=None, workspace: Optional[torch.Tensor] = None,
                            stream=None):
    """``gdn_chunk_prefill`` with per-kernel timing (see
    ``gdn_chunk_prefill_timed`` in include/gdn.h).  ``events``: four
    torch.cuda.Event(enable_timing=True) (created if None), recorded before
    the chunk table, after it, after prep and after the recurrence.  Returns
    (out, final_state, fused, events); read the kernel times with
    events[i].elapsed_time(events[i + 1]) after synchronising."""
    if events is None:
        events = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    if len(events) != 4:
        raise ValueError("events must hold four torch.cuda.Event")
    out, final_state, fused = _prefill(q, k, v, g, beta, cu_seqlens, initial_state, out,
                                       final_state, output_final_state, workspace, stream,
                                       _NO_SNAPSHOTS, 0, events=events)
    return out, final_state, fused, events


def gdn_chunk_prefill_snapshots(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                                g: torch.Tensor, beta: torch.Tensor, cu_seqlens: torch.Tensor,
                                initial_state: Optional[torch.Tensor] = None,
                                out: Optional[torch.Tensor] = None,
                                final_state: Optional[torch.Tensor] = None,
                                output_final_state: bool = False,
                                snapshots: Optional[torch.Tensor] = None,
                                snapshot_chunks: int = 1,
                                workspace: Optional[torch.Tensor] = None, stream=None):
    """``gdn_chunk_prefill`` that also returns states at chunk boundaries (see
    ``gdn_chunk_prefill_snapshots`` in include/gdn.h): one after every
    ``snapshot_chunks`` chunks (64 tokens each) and after the last chunk of
    each sequence.  Returns (out, final_state, snapshots [slots, Hv, dv, dk]
    fp32); sequence n's snapshot i is slot sum_{m<n} ceil(chunks_m / s) + i."""
    return _prefill(q, k, v, g, beta, cu_seqlens, initial_state, out, final_state,
                    output_final_state, workspace, stream, snapshots, snapshot_chunks)


def gdn_chunk_prefill_scan(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                           g: torch.Tensor, beta: torch.Tensor, cu_seqlens: torch.Tensor,
                           initial_state: Optional[torch.Tensor] = None,
                           out: Optional[torch.Tensor] = None,
                           final_state: Optional[torch.Tensor] = None,
                           output_final_state: bool = False, chunks_per_group: int = 0,
                           workspace: Optional[torch.Tensor] = None, stream=None):
    """``gdn_chunk_prefill`` with the chunk recurrence as a chunk-parallel scan
    over groups of ``chunks_per_group`` chunks (0: chosen to fill the SMs);
    see ``gdn_chunk_prefill_scan`` in include/gdn.h.  Returns (out,
    final_state)."""
    return _prefill(q, k, v, g, beta, cu_seqlens, initial_state, out, final_state,
                    output_final_state, workspace, stream, _NO_SNAPSHOTS, 0,
                    scan_group=int(chunks_per_group))


def gdn_chunk_prefill_scan_workspace_size(N: int, T: int, Hk: int, Hv: int, dk: int, dv: int,
                                          chunks_per_group: int = 0,
                                          dtype=torch.bfloat16) -> int:
    """Workspace bytes of ``gdn_chunk_prefill_scan`` (0 if unsupported)."""
    p = make_problem(N, T, Hk, Hv, dk, dv, dtype)
    return int(library().gdn_chunk_prefill_scan_workspace_size(ctypes.byref(p),
                                                                 chunks_per_group))


def gdn_chunk_prefill_device_status(workspace: Optional[torch.Tensor] = None,
                                    stream=None, noalloc: bool = False) -> int:
    """Device-side status of the last bf16 (d = 128) prefill (see
    ``gdn_chunk_prefill_device_status`` in include/gdn.h): waits for the
    stream and returns GDN_OK, GDN_ERR_INVALID_ARG (malformed cu_seqlens),
    GDN_ERR_TIMEOUT (a bounded device wait ran out) or GDN_ERR_CUDA.
    ``workspace``: the one the call used; by default the workspace this
    module keeps for the current device, `stream` and host thread, or with
    ``noalloc`` the built-in
    scratch of ``gdn_chunk_prefill_noalloc``."""
    if noalloc:
        ptr = None
    else:
        if workspace is None:
            workspace = _workspaces.get(
                _workspace_key(torch.device("cuda", torch.cuda.current_device()), stream))
            if workspace is None:
                raise ValueError("no workspace: no prefill has run through this module")
        ptr = workspace.data_ptr()
    return int(library().gdn_chunk_prefill_device_status(ptr, _stream(stream)))


NOALLOC_SCRATCH_BYTES = 64 << 20


def gdn_chunk_prefill_noalloc(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                              g: torch.Tensor, beta: torch.Tensor, cu_seqlens: torch.Tensor,
                              initial_state: Optional[torch.Tensor] = None,
                              out: torch.Tensor = None,
                              final_state: Optional[torch.Tensor] = None,
                              stream=None) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """``gdn_chunk_prefill`` for callers that cannot allocate device memory at
    call time: the library's built-in 64 MiB scratch array replaces the
    workspace, and ``out`` (and ``final_state`` if wanted) must be given, so
    this wrapper allocates nothing either.  Problems needing more than 64 MiB
    of workspace raise GDNError(GDN_ERR_WORKSPACE).  Calls that may overlap on
    the GPU share the scratch and must be ordered by the caller."""
    T, Hk, dk = q.shape
    Hv, dv = v.shape[1], v.shape[2]
    N = cu_seqlens.shape[0] - 1
    dt = q.dtype
    if dt not in _DTYPES:
        raise TypeError(f"unsupported q/k/v dtype {dt}")
    if out is None:
        raise ValueError("gdn_chunk_prefill_noalloc needs a preallocated out")
    for t, name, tdt, shape in ((q, "q", dt, (T, Hk, dk)), (k, "k", dt, (T, Hk, dk)),
                                (v, "v", dt, (T, Hv, dv)), (g, "g", torch.float32, (T, Hv)),
                                (beta, "beta", torch.float32, (T, Hv)),
                                (cu_seqlens, "cu_seqlens", torch.int32, (N + 1,)),
                                (out, "out", dt, (T, Hv, dv))):
        _check(t, name, tdt, shape)
    for t, name in ((initial_state, "initial_state"), (final_state, "final_state")):
        if t is not None:
            _check(t, name, torch.float32, (N, Hv, dv, dk))
    _same_device(q.device, k=k, v=v, g=g, beta=beta, cu_seqlens=cu_seqlens,
                 initial_state=initial_state, out=out, final_state=final_state)
    p = make_problem(N, T, Hk, Hv, dk, dv, dt)
    with torch.cuda.device(q.device):  # the built-in scratch of q's device
        rc = library().gdn_chunk_prefill_noalloc(
            ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu_seqlens),
            _ptr(initial_state), _ptr(out), _ptr(final_state), _stream(stream))
    if rc != 0:
        raise GDNError(rc, "gdn_chunk_prefill_noalloc")
    return out, final_state


def gdn_decode_step(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                    g: torch.Tensor, beta: torch.Tensor, state: torch.Tensor,
                    out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """One recurrent step per sequence, updating ``state`` in place (see
    ``gdn_decode_step`` in include/gdn.h).  q, k: [N, Hk, dk]; v: [N, Hv, dv];
    g, beta: [N, Hv] fp32; state: [N, Hv, dv, dk] fp32.  Returns out [N, Hv, dv]."""
    N, Hk, dk = q.shape
    Hv, dv = v.shape[1], v.shape[2]
    dt = q.dtype
    if dt not in _DTYPES:
        raise TypeError(f"unsupported q/k/v dtype {dt}")
    _check(q, "q", dt, (N, Hk, dk))
    _check(k, "k", dt, (N, Hk, dk))
    _check(v, "v", dt, (N, Hv, dv))
    _check(g, "g", torch.float32, (N, Hv))
    _check(beta, "beta", torch.float32, (N, Hv))
    _check(state, "state", torch.float32, (N, Hv, dv, dk))
    if out is None:
        out = torch.empty((N, Hv, dv), dtype=dt, device=q.device)
    _check(out, "out", dt, (N, Hv, dv))
    _same_device(q.device, k=k, v=v, g=g, beta=beta, state=state, out=out)
    p = make_problem(N, N, Hk, Hv, dk, dv, dt)
    with torch.cuda.device(q.device):
        rc = library().gdn_decode_step(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                       _ptr(beta), _ptr(state), _ptr(out), _stream(stream))
    if rc != 0:
        raise GDNError(rc, "gdn_decode_step")
    return out


_STATE_DTYPES = {torch.float16: GDN_F16, torch.bfloat16: GDN_BF16}


def gdn_decode_step_half_state(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                               g: torch.Tensor, beta: torch.Tensor, state: torch.Tensor,
                               out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """``gdn_decode_step`` with a 16-bit state (fp16 or bf16, updated in place;
    see ``gdn_decode_step_half_state`` in include/gdn.h).  Returns out."""
    N, Hk, dk = q.shape
    Hv, dv = v.shape[1], v.shape[2]
    dt = q.dtype
    if dt not in _DTYPES:
        raise TypeError(f"unsupported q/k/v dtype {dt}")
    if state.dtype not in _STATE_DTYPES:
        raise TypeError(f"state must be float16 or bfloat16, got {state.dtype}")
    _check(q, "q", dt, (N, Hk, dk))
    _check(k, "k", dt, (N, Hk, dk))
    _check(v, "v", dt, (N, Hv, dv))
    _check(g, "g", torch.float32, (N, Hv))
    _check(beta, "beta", torch.float32, (N, Hv))
    _check(state, "state", state.dtype, (N, Hv, dv, dk))
    if out is None:
        out = torch.empty((N, Hv, dv), dtype=dt, device=q.device)
    _check(out, "out", dt, (N, Hv, dv))
    _same_device(q.device, k=k, v=v, g=g, beta=beta, state=state, out=out)
    p = make_problem(N, N, Hk, Hv, dk, dv, dt)
    with torch.cuda.device(q.device):
        rc = library().gdn_decode_step_half_state(
            ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state),
            _STATE_DTYPES[state.dtype], _ptr(out), _stream(stream))
    if rc != 0:
        raise GDNError(rc, "gdn_decode_step_half_state")
    return out


_ALL_STATE_DTYPES = {torch.float32: GDN_F32, torch.float16: GDN_F16, torch.bfloat16: GDN_BF16}


def gdn_verify_step(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor,
                    beta: torch.Tensor, state: torch.Tensor,
                    slots: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                    stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Verify step of speculative decoding (see ``gdn_verify_step`` in
    include/gdn.h).  q, k: [N, K, Hk, dk]; v: [N, K, Hv, dv]; g, beta:
    [N, K, Hv] fp32 (K = 1 .. 8 tokens per sequence); state [N, Hv, dv, dk]
    in fp32, fp16 or bf16 (read only).  Returns (out [N, K, Hv, dv], slots
    [N, K, Hv, dv, dk] in the state's dtype: the state after each token)."""
    N, K, Hk, dk = q.shape
    Hv, dv = v.shape[2], v.shape[3]
    dt = q.dtype
    if dt not in _DTYPES:
        raise TypeError(f"unsupported q/k/v dtype {dt}")
    if state.dtype not in _ALL_STATE_DTYPES:
        raise TypeError(f"unsupported state dtype {state.dtype}")
    _check(q, "q", dt, (N, K, Hk, dk))
    _check(k, "k", dt, (N, K, Hk, dk))
    _check(v, "v", dt, (N, K, Hv, dv))
    _check(g, "g", torch.float32, (N, K, Hv))
    _check(beta, "beta", torch.float32, (N, K, Hv))
    _check(state, "state", state.dtype, (N, Hv, dv, dk))
    if slots is None:
        slots = torch.empty((N, K, Hv, dv, dk), dtype=state.dtype, device=q.device)
    _check(slots, "slots", state.dtype, (N, K, Hv, dv, dk))
    if out is None:
        out = torch.empty((N, K, Hv, dv), dtype=dt, device=q.device)
    _check(out, "out", dt, (N, K, Hv, dv))
    _same_device(q.device, k=k, v=v, g=g, beta=beta, state=state, slots=slots, out=out)
    p = make_problem(N, N * K, Hk, Hv, dk, dv, dt)
    with torch.cuda.device(q.device):
        rc = library().gdn_verify_step(ctypes.byref(p), K, _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                       _ptr(beta), _ptr(state), _ALL_STATE_DTYPES[state.dtype],
                                       _ptr(slots), _ptr(out), _stream(stream))
    if rc != 0:
        raise GDNError(rc, "gdn_verify_step")
    return out, slots


def prefill_launches(Hv: int, d: int, dtype, total_tokens: int = 1) -> int:
    """Kernel launches one gdn_chunk_prefill call makes (for launch counts):
    the tensor-core path (bf16, d = 128) runs the chunk-table, prep and
    recurrence kernels (no prep when there are no tokens); the fp32 path one
    kernel."""
    if dtype == torch.bfloat16 and d == 128:
        return 3 if total_tokens > 0 else 2
    return 1
