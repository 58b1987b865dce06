"""ctypes binding of librsc.so (include/rsc.h) with the same entry-point names.

Argument marshalling only: torch tensors are checked for dtype, device, shape and
contiguity, then their device pointers and the current CUDA stream are handed to the C
ABI.  Every step of the layer runs in the library's CUDA kernels; there is no fallback
of any kind, and a missing library raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _build

F32, BF16 = 0, 1
KDA, GDN = 0, 1
VERIFY, COMMIT = 0, 1

RSC_OK, RSC_EINVAL, RSC_ERANGE, RSC_EDTYPE, RSC_EALIGN, RSC_ECUDA, RSC_ENOSPACE, RSC_EDEVICE = (
    0, -1, -2, -3, -4, -5, -6, -7)
DEVERR_SLOT, DEVERR_ACCEPT, DEVERR_SEQ, DEVERR_TIMEOUT, DEVERR_GATE, DEVERR_RING = 1, 2, 4, 8, 16, 32

TORCH_DTYPE = {F32: torch.float32, BF16: torch.bfloat16}

# Every symbol include/rsc.h declares.
EXPORTS = ("ssm_pool_create", "ssm_pool_destroy", "ssm_pool_bytes", "kda_decode_step",
           "kda_decode_step_overlap", "kda_decode_step_ex", "kda_decode_step_gated",
           "kda_decode_step_track",
           "kda_prefill_workspace_size", "kda_prefill_chunk", "kda_prefill_chunk_noalloc",
           "ssm_slot_copy",
           "kda_spec_verify_commit", "kda_replay_verify_commit", "rsc_get_device_error",
           "rsc_status_string", "rsc_slot_alloc_create", "rsc_slot_alloc_destroy",
           "rsc_slot_alloc_free_count", "rsc_slot_alloc_acquire", "rsc_slot_alloc_release",
           "rsc_max_running_requests", "rsc_track_plan")


class RscError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status} ({status_string(status)})")


class PoolDesc(ctypes.Structure):
    _fields_ = [
        ("num_layers", ctypes.c_int32), ("num_slots", ctypes.c_int32),
        ("num_heads", ctypes.c_int32), ("head_k", ctypes.c_int32),
        ("head_v", ctypes.c_int32), ("conv_kernel", ctypes.c_int32),
        ("state_dtype", ctypes.c_int32), ("conv_dtype", ctypes.c_int32),
        ("gate", ctypes.c_int32),
        ("ssm_base", ctypes.c_void_p), ("conv_base", ctypes.c_void_p),
        ("dev_error", ctypes.c_void_p),
    ]


class DecodeOpts(ctypes.Structure):
    """rsc_decode_opts of include/rsc.h."""
    _fields_ = [
        ("A_log", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p),
        ("track_mask", ctypes.c_void_p), ("track_slots", ctypes.c_void_p),
        ("flags", ctypes.c_int32),
    ]


DECODE_OVERLAP = 1


class ReplayRingsDesc(ctypes.Structure):
    _fields_ = [
        ("depth", ctypes.c_int32),
        ("d", ctypes.c_void_p), ("k", ctypes.c_void_p), ("rawv", ctypes.c_void_p),
        ("rawk", ctypes.c_void_p), ("g", ctypes.c_void_p), ("beta", ctypes.c_void_p),
    ]


_lib = None


def library_path() -> str:
    return _build.LIB


def lib():
    """The loaded librsc.so.  Raises if it has not been built (no fallback exists)."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"librsc.so is missing at {path}: build it with "
                               "recurrent_state_cache_gb300._build.build()")
        L = ctypes.CDLL(path)
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        pd = ctypes.POINTER(PoolDesc)
        L.ssm_pool_create.argtypes = [pd, ctypes.POINTER(vp)]
        L.ssm_pool_destroy.argtypes = [vp]
        L.ssm_pool_bytes.argtypes = [pd, ctypes.POINTER(ctypes.c_uint64),
                                     ctypes.POINTER(ctypes.c_uint64)]
        L.kda_decode_step.argtypes = [vp, i32, vp, i32, vp, vp, vp, vp, vp, vp]
        L.kda_decode_step_overlap.argtypes = [vp, i32, vp, i32, vp, vp, vp, vp, vp, vp]
        L.kda_decode_step_ex.argtypes = [vp, i32, vp, i32, vp, vp, vp, vp, vp, vp, vp]
        L.kda_decode_step_track.argtypes = [vp, i32, vp, i32, vp, vp, vp, vp, vp, vp, vp, vp]
        L.kda_decode_step_gated.argtypes = [vp, i32, vp, i32, vp, vp, vp, vp, vp, vp, vp, vp]
        L.kda_prefill_workspace_size.argtypes = [vp, i32, i32, ctypes.POINTER(sz)]
        L.kda_prefill_chunk.argtypes = [vp, i32, vp, vp, i32, i32, vp, vp, vp, vp, vp, vp,
                                        vp, sz, vp]
        L.kda_prefill_chunk_noalloc.argtypes = [vp, i32, vp, vp, i32, i32, vp, vp, vp, vp, vp,
                                                vp, vp]
        L.ssm_slot_copy.argtypes = [vp, i32, vp, vp, vp, i32, vp]
        L.kda_spec_verify_commit.argtypes = [vp, i32, i32, vp, i32, i32, i32, vp, vp, vp, vp,
                                             vp, vp, vp, vp, vp]
        L.kda_replay_verify_commit.argtypes = [vp, ctypes.POINTER(ReplayRingsDesc), i32, i32,
                                               vp, vp, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp]
        L.rsc_get_device_error.argtypes = [vp, ctypes.POINTER(ctypes.c_int32), vp]
        ip = ctypes.POINTER(ctypes.c_int)
        L.rsc_slot_alloc_create.argtypes = [i32, ctypes.POINTER(vp)]
        L.rsc_slot_alloc_destroy.argtypes = [vp]
        L.rsc_slot_alloc_free_count.argtypes = [vp, ip]
        L.rsc_slot_alloc_acquire.argtypes = [vp, i32, vp]
        L.rsc_slot_alloc_release.argtypes = [vp, i32, vp]
        L.rsc_max_running_requests.argtypes = [i32, i32, i32, ip]
        L.rsc_track_plan.argtypes = [i32, vp, i32, vp, i32, vp, vp, vp]
        L.rsc_status_string.argtypes = [i32]
        L.rsc_status_string.restype = ctypes.c_char_p
        for name in EXPORTS:
            if name != "rsc_status_string":
                getattr(L, name).restype = i32
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().rsc_status_string(status).decode()


def _check(rc: int, what: str):
    if rc != RSC_OK:
        raise RscError(rc, what)


# The per-call marshalling below runs once per library call, so it keeps to cheap operations:
# raw pointers and stream handles as plain ints (the argtypes convert them), device checks by
# index.  Every check of the argument still happens.

def _p(t):
    return None if t is None else t.data_ptr()


# torch's current stream of a device as its raw handle, without building a Stream object
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream, pool):
    """The call's stream (raw handle): `stream`, else the current torch stream of the pool's
    device."""
    if stream is None:
        if _raw_stream is not None:
            return _raw_stream(pool.device.index)
        stream = torch.cuda.current_stream(pool.device)
    if stream.device != pool.device:
        raise ValueError(f"stream on {stream.device}, the pool is on {pool.device}")
    return stream.cuda_stream


class _on:
    """Makes the pool's device current for one library call (the library launches on the
    current device and rejects a pool held by another one)."""

    __slots__ = ("dev", "prev")

    def __init__(self, pool):
        self.dev = pool.device.index
        self.prev = None

    def __enter__(self):
        cur = torch.cuda.current_device()
        if cur != self.dev:
            self.prev = cur
            torch.cuda.set_device(self.dev)

    def __exit__(self, *exc):
        if self.prev is not None:
            torch.cuda.set_device(self.prev)


def _need(t, name, dtype, shape, device):
    if t.dtype is not dtype:
        raise ValueError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if t.get_device() != device.index:
        raise ValueError(f"{name}: on {t.device}, expected {device}")
    if t.shape != shape:
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")


class SlotPool:
    """A slot pool in device memory allocated by torch, plus the library's host handle.

    ssm  [num_layers][num_slots+1][H][V][K]  state dtype
    conv [num_layers][num_slots+1][3][D]     conv dtype (also the io dtype)
    """

    def __init__(self, num_layers, num_slots, H, K, V, state_dtype=BF16, conv_dtype=BF16,
                 gate=KDA, device="cuda", ssm=None, conv=None):
        self.device = torch.device(device)
        if self.device.type == "cuda" and self.device.index is None:
            self.device = torch.device("cuda", torch.cuda.current_device())
        self.num_layers, self.num_slots = num_layers, num_slots
        self.H, self.K, self.V = H, K, V
        self.D = H * (2 * K + V)
        self.state_dtype, self.conv_dtype, self.gate = state_dtype, conv_dtype, gate
        rows = num_slots + 1
        shp_s, shp_c = (num_layers, rows, H, V, K), (num_layers, rows, 3, self.D)
        self.ssm = (torch.zeros(shp_s, dtype=TORCH_DTYPE[state_dtype], device=self.device)
                    if ssm is None else ssm)
        self.conv = (torch.zeros(shp_c, dtype=TORCH_DTYPE[conv_dtype], device=self.device)
                     if conv is None else conv)
        _need(self.ssm, "ssm", TORCH_DTYPE[state_dtype], shp_s, self.device)
        _need(self.conv, "conv", TORCH_DTYPE[conv_dtype], shp_c, self.device)
        self.dev_error = torch.zeros(4, dtype=torch.int32, device=self.device)
        self.desc = PoolDesc(num_layers, num_slots, H, K, V, 4, state_dtype, conv_dtype, gate,
                             self.ssm.data_ptr(), self.conv.data_ptr(),
                             self.dev_error.data_ptr())
        h = ctypes.c_void_p()
        _check(lib().ssm_pool_create(ctypes.byref(self.desc), ctypes.byref(h)),
               "ssm_pool_create")
        self.handle = h

    def close(self):
        if getattr(self, "handle", None):
            lib().ssm_pool_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def io_dtype(self):
        return TORCH_DTYPE[self.conv_dtype]

    def gate_shape(self, lead):
        return tuple(lead) + ((self.H, self.K) if self.gate == KDA else (self.H,))


def ssm_pool_bytes(num_layers, num_slots, H, K, V, state_dtype, conv_dtype, gate=KDA):
    d = PoolDesc(num_layers, num_slots, H, K, V, 4, state_dtype, conv_dtype, gate, None, None,
                 None)
    s, c = ctypes.c_uint64(), ctypes.c_uint64()
    _check(lib().ssm_pool_bytes(ctypes.byref(d), ctypes.byref(s), ctypes.byref(c)),
           "ssm_pool_bytes")
    return s.value, c.value


def kda_decode_step(pool: SlotPool, layer, slot_ids, qkv, conv_w, g, beta, out=None,
                    stream=None, overlap=False):
    """One decode step of layer `layer` for the requests in slot_ids.  overlap=True calls
    kda_decode_step_overlap: the kernel reads slot_ids and this layer's state and window
    rows of those slots before the earlier kernels on the stream finish, so none of them
    may write those (see include/rsc.h)."""
    B = slot_ids.shape[0]
    dev = pool.device
    _need(slot_ids, "slot_ids", torch.int32, (B,), dev)
    _need(qkv, "qkv", pool.io_dtype, (B, pool.D), dev)
    _need(conv_w, "conv_w", torch.float32, (pool.D, 4), dev)
    _need(g, "g", torch.float32, pool.gate_shape((B,)), dev)
    _need(beta, "beta", torch.float32, (B, pool.H), dev)
    if out is None:
        out = torch.empty((B, pool.H, pool.V), dtype=pool.io_dtype, device=dev)
    _need(out, "out", pool.io_dtype, (B, pool.H, pool.V), dev)
    fn = lib().kda_decode_step_overlap if overlap else lib().kda_decode_step
    with _on(pool):
        _check(fn(pool.handle, layer, _p(slot_ids), B, _p(qkv), _p(conv_w), _p(g), _p(beta),
                  _p(out), _stream(stream, pool)),
               "kda_decode_step_overlap" if overlap else "kda_decode_step")
    return out


def kda_prefill_workspace_size(pool: SlotPool, num_seqs, total_tokens) -> int:
    n = ctypes.c_size_t()
    _check(lib().kda_prefill_workspace_size(pool.handle, num_seqs, total_tokens,
                                            ctypes.byref(n)), "kda_prefill_workspace_size")
    return n.value


def kda_prefill_chunk(pool: SlotPool, layer, slot_ids, cu_seqlens, qkv, conv_w, g, beta,
                      has_initial_state=None, out=None, workspace=None, stream=None):
    N = slot_ids.shape[0]
    T = qkv.shape[0]
    dev = pool.device
    _need(slot_ids, "slot_ids", torch.int32, (N,), dev)
    _need(cu_seqlens, "cu_seqlens", torch.int32, (N + 1,), dev)
    _need(qkv, "qkv", pool.io_dtype, (T, pool.D), dev)
    _need(conv_w, "conv_w", torch.float32, (pool.D, 4), dev)
    _need(g, "g", torch.float32, pool.gate_shape((T,)), dev)
    _need(beta, "beta", torch.float32, (T, pool.H), dev)
    if has_initial_state is not None:
        _need(has_initial_state, "has_initial_state", torch.uint8, (N,), dev)
    if out is None:
        out = torch.empty((T, pool.H, pool.V), dtype=pool.io_dtype, device=dev)
    _need(out, "out", pool.io_dtype, (T, pool.H, pool.V), dev)
    need = kda_prefill_workspace_size(pool, N, T)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    if workspace.dtype != torch.uint8 or workspace.device != dev:
        raise ValueError("workspace: a uint8 tensor on the pool's device")
    with _on(pool):
        _check(lib().kda_prefill_chunk(pool.handle, layer, _p(slot_ids), _p(cu_seqlens), N, T,
                                       _p(has_initial_state), _p(qkv), _p(conv_w), _p(g), _p(beta),
                                       _p(out), _p(workspace), workspace.numel(), _stream(stream, pool)),
               "kda_prefill_chunk")
    return out


def kda_prefill_chunk_noalloc(pool: SlotPool, layer, slot_ids, cu_seqlens, qkv, conv_w, g,
                              beta, has_initial_state=None, out=None, stream=None):
    """kda_prefill_chunk on the library's static device scratch, for callers that cannot
    allocate device memory (all of HBM already given to their own pools, or no
    tolerance for cudaMalloc's device synchronisation).  Allocates nothing besides
    `out` when it is not given.  Calls share the scratch: keep them on one stream."""
    N = slot_ids.shape[0]
    T = qkv.shape[0]
    dev = pool.device
    _need(slot_ids, "slot_ids", torch.int32, (N,), dev)
    _need(cu_seqlens, "cu_seqlens", torch.int32, (N + 1,), dev)
    _need(qkv, "qkv", pool.io_dtype, (T, pool.D), dev)
    _need(conv_w, "conv_w", torch.float32, (pool.D, 4), dev)
    _need(g, "g", torch.float32, pool.gate_shape((T,)), dev)
    _need(beta, "beta", torch.float32, (T, pool.H), dev)
    if has_initial_state is not None:
        _need(has_initial_state, "has_initial_state", torch.uint8, (N,), dev)
    if out is None:
        out = torch.empty((T, pool.H, pool.V), dtype=pool.io_dtype, device=dev)
    _need(out, "out", pool.io_dtype, (T, pool.H, pool.V), dev)
    with _on(pool):
        _check(lib().kda_prefill_chunk_noalloc(pool.handle, layer, _p(slot_ids), _p(cu_seqlens), N,
                                               T, _p(has_initial_state), _p(qkv), _p(conv_w), _p(g),
                                               _p(beta), _p(out), _stream(stream, pool)),
               "kda_prefill_chunk_noalloc")
    return out


def kda_decode_step_ex(pool: SlotPool, layer, slot_ids, qkv, conv_w, g, beta, out=None,
                       A_log=None, dt_bias=None, track_mask=None, track_slots=None,
                       overlap=False, stream=None):
    """The general decode call (kda_decode_step_ex): any combination of fused gating (A_log,
    dt_bias given; g and beta are then the raw projections a and b), the fused track copy
    (track_mask, track_slots given) and the overlapped launch."""
    B = slot_ids.shape[0]
    dev = pool.device
    _need(slot_ids, "slot_ids", torch.int32, (B,), dev)
    _need(qkv, "qkv", pool.io_dtype, (B, pool.D), dev)
    _need(conv_w, "conv_w", torch.float32, (pool.D, 4), dev)
    _need(g, "g", torch.float32, pool.gate_shape((B,)), dev)
    _need(beta, "beta", torch.float32, (B, pool.H), dev)
    if A_log is not None or dt_bias is not None:
        n = pool.K if pool.gate == KDA else 1
        _need(A_log, "A_log", torch.float32, (pool.H,), dev)
        _need(dt_bias, "dt_bias", torch.float32, (pool.H, n) if n > 1 else (pool.H,), dev)
    if track_mask is not None or track_slots is not None:
        _need(track_mask, "track_mask", torch.uint8, (B,), dev)
        _need(track_slots, "track_slots", torch.int32, (B,), dev)
    if out is None:
        out = torch.empty((B, pool.H, pool.V), dtype=pool.io_dtype, device=dev)
    _need(out, "out", pool.io_dtype, (B, pool.H, pool.V), dev)
    addr = lambda t: None if t is None else t.data_ptr()
    opts = DecodeOpts(addr(A_log), addr(dt_bias), addr(track_mask), addr(track_slots),
                      DECODE_OVERLAP if overlap else 0)
    with _on(pool):
        _check(lib().kda_decode_step_ex(pool.handle, layer, _p(slot_ids), B, _p(qkv), _p(conv_w),
                                        _p(g), _p(beta), _p(out), ctypes.byref(opts),
                                        _stream(stream, pool)), "kda_decode_step_ex")
    return out


def kda_decode_step_track(pool: SlotPool, layer, slot_ids, qkv, conv_w, g, beta, track_mask,
                          track_slots, out=None, stream=None):
    """Decode, and for requests with track_mask set the updated state and window written
    into track_slots as well (the masked track copy, fused)."""
    B = slot_ids.shape[0]
    dev = pool.device
    _need(slot_ids, "slot_ids", torch.int32, (B,), dev)
    _need(qkv, "qkv", pool.io_dtype, (B, pool.D), dev)
    _need(conv_w, "conv_w", torch.float32, (pool.D, 4), dev)
    _need(g, "g", torch.float32, pool.gate_shape((B,)), dev)
    _need(beta, "beta", torch.float32, (B, pool.H), dev)
    _need(track_mask, "track_mask", torch.uint8, (B,), dev)
    _need(track_slots, "track_slots", torch.int32, (B,), dev)
    if out is None:
        out = torch.empty((B, pool.H, pool.V), dtype=pool.io_dtype, device=dev)
    _need(out, "out", pool.io_dtype, (B, pool.H, pool.V), dev)
    with _on(pool):
        _check(lib().kda_decode_step_track(pool.handle, layer, _p(slot_ids), B, _p(qkv), _p(conv_w),
                                           _p(g), _p(beta), _p(out), _p(track_mask), _p(track_slots),
                                           _stream(stream, pool)), "kda_decode_step_track")
    return out


def kda_decode_step_gated(pool: SlotPool, layer, slot_ids, qkv, conv_w, a, b, A_log, dt_bias,
                          out=None, stream=None):
    """Decode with the gates formed in the kernel from the raw projections a, b (see the
    header for the gating reading)."""
    B = slot_ids.shape[0]
    dev = pool.device
    n = pool.K if pool.gate == KDA else 1
    _need(slot_ids, "slot_ids", torch.int32, (B,), dev)
    _need(qkv, "qkv", pool.io_dtype, (B, pool.D), dev)
    _need(conv_w, "conv_w", torch.float32, (pool.D, 4), dev)
    _need(a, "a", torch.float32, pool.gate_shape((B,)), dev)
    _need(b, "b", torch.float32, (B, pool.H), dev)
    _need(A_log, "A_log", torch.float32, (pool.H,), dev)
    _need(dt_bias, "dt_bias", torch.float32, (pool.H, n) if n > 1 else (pool.H,), dev)
    if out is None:
        out = torch.empty((B, pool.H, pool.V), dtype=pool.io_dtype, device=dev)
    _need(out, "out", pool.io_dtype, (B, pool.H, pool.V), dev)
    with _on(pool):
        _check(lib().kda_decode_step_gated(pool.handle, layer, _p(slot_ids), B, _p(qkv), _p(conv_w),
                                           _p(a), _p(b), _p(A_log), _p(dt_bias), _p(out),
                                           _stream(stream, pool)), "kda_decode_step_gated")
    return out


def ssm_slot_copy(pool: SlotPool, layer, src, dst, mask=None, stream=None):
    n = src.shape[0]
    dev = pool.device
    _need(src, "src", torch.int32, (n,), dev)
    _need(dst, "dst", torch.int32, (n,), dev)
    if mask is not None:
        _need(mask, "mask", torch.uint8, (n,), dev)
    with _on(pool):
        _check(lib().ssm_slot_copy(pool.handle, layer, _p(src), _p(dst), _p(mask), n,
                                   _stream(stream, pool)), "ssm_slot_copy")


def kda_spec_verify_commit(pool: SlotPool, layer, mode, slot_ids, T, L, spec_ssm, spec_conv,
                           qkv=None, conv_w=None, g=None, beta=None, out=None, accept=None,
                           stream=None):
    B = slot_ids.shape[0]
    dev = pool.device
    _need(slot_ids, "slot_ids", torch.int32, (B,), dev)
    _need(spec_ssm, "spec_ssm", TORCH_DTYPE[pool.state_dtype], (B, L, pool.H, pool.V, pool.K), dev)
    _need(spec_conv, "spec_conv", pool.io_dtype, (B, L, 3, pool.D), dev)
    if mode == VERIFY:
        _need(qkv, "qkv", pool.io_dtype, (B, T, pool.D), dev)
        _need(conv_w, "conv_w", torch.float32, (pool.D, 4), dev)
        _need(g, "g", torch.float32, pool.gate_shape((B, T)), dev)
        _need(beta, "beta", torch.float32, (B, T, pool.H), dev)
        if out is None:
            out = torch.empty((B, T, pool.H, pool.V), dtype=pool.io_dtype, device=dev)
        _need(out, "out", pool.io_dtype, (B, T, pool.H, pool.V), dev)
    else:
        _need(accept, "accept", torch.int32, (B,), dev)
    with _on(pool):
        _check(lib().kda_spec_verify_commit(pool.handle, layer, mode, _p(slot_ids), B, T, L,
                                            _p(spec_ssm), _p(spec_conv), _p(qkv), _p(conv_w), _p(g),
                                            _p(beta), _p(out), _p(accept), _stream(stream, pool)),
               "kda_spec_verify_commit")
    return out


class ReplayRings:
    """ReplaySSM rings of a pool, allocated by torch ([layers][slots+1][H][depth][n]):
    d, rawv [..][V] and k, rawk [..][K] in the state dtype; g [..][K] (KDA) or [..] (GDN)
    and beta [..] in fp32."""

    def __init__(self, pool: SlotPool, depth: int):
        L, R, H, K, V = pool.num_layers, pool.num_slots + 1, pool.H, pool.K, pool.V
        sd, dev = TORCH_DTYPE[pool.state_dtype], pool.device
        self.depth = depth
        self.d = torch.zeros((L, R, H, depth, V), dtype=sd, device=dev)
        self.k = torch.zeros((L, R, H, depth, K), dtype=sd, device=dev)
        self.rawv = torch.zeros((L, R, H, depth, V), dtype=sd, device=dev)
        self.rawk = torch.zeros((L, R, H, depth, K), dtype=sd, device=dev)
        gshape = (L, R, H, depth, K) if pool.gate == KDA else (L, R, H, depth)
        self.g = torch.zeros(gshape, dtype=torch.float32, device=dev)
        self.beta = torch.zeros((L, R, H, depth), dtype=torch.float32, device=dev)

    def desc(self) -> ReplayRingsDesc:
        return ReplayRingsDesc(self.depth, self.d.data_ptr(), self.k.data_ptr(),
                               self.rawv.data_ptr(), self.rawk.data_ptr(), self.g.data_ptr(),
                               self.beta.data_ptr())


def kda_replay_verify_commit(pool: SlotPool, rings: ReplayRings, layer, mode, slot_ids, ring_pos,
                             T, spec_conv, qkv=None, conv_w=None, g=None, beta=None, out=None,
                             accept=None, stream=None):
    B = slot_ids.shape[0]
    dev = pool.device
    _need(slot_ids, "slot_ids", torch.int32, (B,), dev)
    _need(ring_pos, "ring_pos", torch.int32, (B,), dev)
    _need(spec_conv, "spec_conv", pool.io_dtype, (B, rings.depth, 3, pool.D), dev)
    if mode == VERIFY:
        _need(qkv, "qkv", pool.io_dtype, (B, T, pool.D), dev)
        _need(conv_w, "conv_w", torch.float32, (pool.D, 4), dev)
        _need(g, "g", torch.float32, pool.gate_shape((B, T)), dev)
        _need(beta, "beta", torch.float32, (B, T, pool.H), dev)
        if out is None:
            out = torch.empty((B, T, pool.H, pool.V), dtype=pool.io_dtype, device=dev)
        _need(out, "out", pool.io_dtype, (B, T, pool.H, pool.V), dev)
    else:
        _need(accept, "accept", torch.int32, (B,), dev)
    d = rings.desc()
    with _on(pool):
        _check(lib().kda_replay_verify_commit(pool.handle, ctypes.byref(d), layer, mode,
                                              _p(slot_ids), _p(ring_pos), B, T, _p(spec_conv),
                                              _p(qkv), _p(conv_w), _p(g), _p(beta), _p(out),
                                              _p(accept), _stream(stream, pool)),
               "kda_replay_verify_commit")
    return out


class SlotAllocator:
    """Host slot allocator of a pool (rsc_slot_alloc): slots 1..num_slots, row 0 never handed
    out.  acquire / release take and give back numpy int32 arrays of slot ids."""

    def __init__(self, num_slots: int):
        import numpy as np
        self._np = np
        h = ctypes.c_void_p()
        _check(lib().rsc_slot_alloc_create(num_slots, ctypes.byref(h)), "rsc_slot_alloc_create")
        self.handle = h
        self.num_slots = num_slots

    def free_count(self) -> int:
        c = ctypes.c_int()
        _check(lib().rsc_slot_alloc_free_count(self.handle, ctypes.byref(c)), "rsc_slot_alloc_free_count")
        return c.value

    def acquire(self, n: int):
        out = self._np.zeros(n, self._np.int32)
        _check(lib().rsc_slot_alloc_acquire(self.handle, n, out.ctypes.data_as(ctypes.c_void_p)),
               "rsc_slot_alloc_acquire")
        return out

    def release(self, slots):
        a = self._np.ascontiguousarray(slots, self._np.int32)
        _check(lib().rsc_slot_alloc_release(self.handle, a.size, a.ctypes.data_as(ctypes.c_void_p)),
               "rsc_slot_alloc_release")

    def __del__(self):
        h = getattr(self, "handle", None)
        if h is not None and h.value and _lib is not None:
            _lib.rsc_slot_alloc_destroy(h)
            self.handle = None


def max_running_requests(num_slots: int, overlap: bool = True, skip_decode_lock: bool = False) -> int:
    c = ctypes.c_int()
    _check(lib().rsc_max_running_requests(num_slots, int(overlap), int(skip_decode_lock),
                                          ctypes.byref(c)), "rsc_max_running_requests")
    return c.value


def track_plan(seq_lens, interval: int, track_pairs, next_idx):
    """(mask uint8 [B], track_slots int32 [B]) of one decode step; next_idx (int32 [B], numpy) is
    advanced in place for the tracked requests."""
    import numpy as np
    sl = np.ascontiguousarray(seq_lens, np.int32)
    tp = np.ascontiguousarray(track_pairs, np.int32)
    B = sl.size
    ntrack = tp.size // max(B, 1)
    assert next_idx.dtype == np.int32 and next_idx.flags["C_CONTIGUOUS"] and next_idx.size == B
    mask = np.zeros(B, np.uint8)
    ts = np.zeros(B, np.int32)
    vp = ctypes.c_void_p
    _check(lib().rsc_track_plan(B, sl.ctypes.data_as(vp), interval, tp.ctypes.data_as(vp), ntrack,
                                next_idx.ctypes.data_as(vp), mask.ctypes.data_as(vp),
                                ts.ctypes.data_as(vp)), "rsc_track_plan")
    return mask, ts


def rsc_get_device_error(pool: SlotPool, stream=None) -> int:
    code = ctypes.c_int32()
    with _on(pool):
        _check(lib().rsc_get_device_error(pool.handle, ctypes.byref(code), _stream(stream, pool)),
               "rsc_get_device_error")
    return code.value
