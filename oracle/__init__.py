"""CPU oracle of the slot-indexed recurrent-state layer step (fp64, plain C).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this package.  The product path
(``recurrent_state_cache_gb300``) never imports, links or calls it, and the two share
no code: this wrapper loads ``rsc_oracle.c`` compiled by gcc, nothing else.

Storage arrays are numpy: fp32 storage as ``np.float32``, bf16 storage as the raw bit
patterns in ``np.uint16``.  Every function mirrors one operation of the pages' method;
the C file cites the passage each one follows.

Pinning status (what the tests check each function against, besides itself):
  conv_sequence      numpy.correlate (a library FIR), window = last three inputs
  recurrent_head     beta=0/alpha=1 identity, single-token closed form, delta-rule write,
                     brute-force product unroll on tiny inputs, the pages' unrolled form
  chunkwise_head     equals recurrent_head (two independent derivations)
  decode/prefill     split order and L2 norm pinned through closed-form special cases
  slot_copy/commit   byte equality
  softplus/sigmoid   values at 0, asymptotes, symmetry; fused-gate decode = decode with them
  replay_verify/     commit(a) equals the snapshot path's commit(a) (fp32 records); the
  replay_commit      records rebuild the state by the pages' closed form; ring wrap-around
  pool_bytes         every logged pool size printed on the pages (tests/golden)
  bf16_round         torch's float32 -> bfloat16 conversion (round to nearest even)
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

F32, BF16 = 0, 1
KDA, GDN = 0, 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rsc_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (IEEE semantics: no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.run(
            ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
             "-o", tmp, _SRC, "-lm"],
            check=True,
        )
        os.replace(tmp, _SO)
    return _SO


class _Rings(ctypes.Structure):
    _fields_ = [
        ("depth", ctypes.c_int32),
        ("d", ctypes.c_void_p), ("k", ctypes.c_void_p), ("rawv", ctypes.c_void_p),
        ("rawk", ctypes.c_void_p), ("g", ctypes.c_void_p), ("beta", ctypes.c_void_p),
    ]


class _Pool(ctypes.Structure):
    _fields_ = [
        ("num_layers", ctypes.c_int32), ("num_slots", ctypes.c_int32),
        ("H", ctypes.c_int32), ("K", ctypes.c_int32), ("V", ctypes.c_int32),
        ("state_dtype", ctypes.c_int32), ("conv_dtype", ctypes.c_int32),
        ("gate", ctypes.c_int32),
        ("ssm", ctypes.c_void_p), ("conv", ctypes.c_void_p),
    ]


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        vp, i32 = ctypes.c_void_p, ctypes.c_int
        pp = ctypes.POINTER(_Pool)
        lib.orc_bf16_round_array.argtypes = [vp, vp, ctypes.c_size_t]
        lib.orc_bf16_round_array.restype = None
        lib.orc_conv_sequence.argtypes = [i32, i32, vp, vp, vp, vp]
        lib.orc_conv_sequence.restype = None
        lib.orc_recurrent_head.argtypes = [i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp]
        lib.orc_recurrent_head.restype = None
        lib.orc_chunkwise_head.argtypes = [i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp]
        lib.orc_chunkwise_head.restype = i32
        lib.orc_pool_bytes.argtypes = [pp, vp, vp]
        lib.orc_pool_bytes.restype = None
        lib.orc_decode_step.argtypes = [pp, i32, vp, i32, vp, vp, vp, vp, vp]
        lib.orc_decode_step.restype = i32
        lib.orc_prefill.argtypes = [pp, i32, vp, vp, i32, vp, vp, vp, vp, vp, vp]
        lib.orc_prefill.restype = i32
        lib.orc_slot_copy.argtypes = [pp, i32, vp, vp, vp, i32]
        lib.orc_slot_copy.restype = i32
        lib.orc_spec_verify.argtypes = [pp, i32, vp, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp]
        lib.orc_spec_verify.restype = i32
        lib.orc_spec_commit.argtypes = [pp, i32, vp, i32, i32, i32, vp, vp, vp]
        lib.orc_spec_commit.restype = i32
        dbl = ctypes.c_double
        lib.orc_softplus.argtypes = [dbl]
        lib.orc_softplus.restype = dbl
        lib.orc_sigmoid.argtypes = [dbl]
        lib.orc_sigmoid.restype = dbl
        lib.orc_gates_from_raw.argtypes = [i32, i32, i32, i32, vp, vp, vp, vp, vp, vp]
        lib.orc_gates_from_raw.restype = None
        lib.orc_decode_step_gated.argtypes = [pp, i32, vp, i32, vp, vp, vp, vp, vp, vp, vp]
        lib.orc_decode_step_gated.restype = i32
        lib.orc_decode_step_track.argtypes = [pp, i32, vp, i32, vp, vp, vp, vp, vp, vp, vp]
        lib.orc_decode_step_track.restype = i32
        rp = ctypes.POINTER(_Rings)
        lib.orc_replay_verify.argtypes = [pp, rp, i32, vp, vp, i32, i32, i32, vp, vp, vp, vp, vp, vp]
        lib.orc_replay_verify.restype = i32
        lib.orc_replay_commit.argtypes = [pp, rp, i32, vp, vp, i32, i32, i32, vp, vp]
        lib.orc_replay_commit.restype = i32
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def storage_np_dtype(dt: int):
    return np.float32 if dt == F32 else np.uint16


# ----------------------------------------------------------------------------- dtypes

def bf16_round(x) -> np.ndarray:
    """Round doubles to bf16 (nearest, ties to even); returns the uint16 bit patterns."""
    x = _c(x, np.float64)
    out = np.empty(x.shape, np.uint16)
    _load().orc_bf16_round_array(_ptr(x), _ptr(out), x.size)
    return out


def bf16_to_f64(bits) -> np.ndarray:
    b = _c(bits, np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def to_f64(a, dt: int) -> np.ndarray:
    return bf16_to_f64(a) if dt == BF16 else np.asarray(a, np.float64)


# ----------------------------------------------------------------------------- pool

class Pool:
    """Host copy of a slot pool: ssm [layers][P+1][H][V][K], conv [layers][P+1][3][D]."""

    def __init__(self, num_layers, num_slots, H, K, V, state_dtype, conv_dtype, gate,
                 ssm=None, conv=None):
        self.num_layers, self.num_slots = num_layers, num_slots
        self.H, self.K, self.V = H, K, V
        self.D = H * (2 * K + V)
        self.state_dtype, self.conv_dtype, self.gate = state_dtype, conv_dtype, gate
        rows = num_slots + 1
        shp_s = (num_layers, rows, H, V, K)
        shp_c = (num_layers, rows, 3, self.D)
        self.ssm = (np.zeros(shp_s, storage_np_dtype(state_dtype)) if ssm is None
                    else _c(ssm, storage_np_dtype(state_dtype)).reshape(shp_s).copy())
        self.conv = (np.zeros(shp_c, storage_np_dtype(conv_dtype)) if conv is None
                     else _c(conv, storage_np_dtype(conv_dtype)).reshape(shp_c).copy())

    def _struct(self):
        return _Pool(self.num_layers, self.num_slots, self.H, self.K, self.V,
                     self.state_dtype, self.conv_dtype, self.gate,
                     self.ssm.ctypes.data, self.conv.ctypes.data)

    def bytes(self):
        s, c = ctypes.c_uint64(), ctypes.c_uint64()
        st = self._struct()
        _load().orc_pool_bytes(ctypes.byref(st), ctypes.byref(s), ctypes.byref(c))
        return s.value, c.value

    def io_np(self):
        return storage_np_dtype(self.conv_dtype)

    def gate_width(self):
        return self.K if self.gate == KDA else 1


def pool_bytes(num_layers, num_slots, H, K, V, state_dtype, conv_dtype):
    """Bytes of the ssm and conv arrays of a pool (without allocating it)."""
    st = _Pool(num_layers, num_slots, H, K, V, state_dtype, conv_dtype, KDA, None, None)
    s, c = ctypes.c_uint64(), ctypes.c_uint64()
    _load().orc_pool_bytes(ctypes.byref(st), ctypes.byref(s), ctypes.byref(c))
    return s.value, c.value


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (rc={rc})")


def _gate_arr(pool, g, lead):
    g = _c(g, np.float32)
    want = lead + ((pool.H, pool.K) if pool.gate == KDA else (pool.H,))
    return g.reshape(want)


def decode_step(pool: Pool, layer, slots, qkv, conv_w, g, beta):
    """One decode token per request; pool updated in place; returns out [B][H][V]."""
    slots = _c(slots, np.int32)
    B = slots.shape[0]
    qkv = _c(qkv, pool.io_np()).reshape(B, pool.D)
    g = _gate_arr(pool, g, (B,))
    beta = _c(beta, np.float32).reshape(B, pool.H)
    w = _c(conv_w, np.float32).reshape(pool.D, 4)
    out = np.zeros((B, pool.H, pool.V), pool.io_np())
    st = pool._struct()
    _check(_load().orc_decode_step(ctypes.byref(st), layer, _ptr(slots), B, _ptr(qkv),
                                   _ptr(w), _ptr(g), _ptr(beta), _ptr(out)), "decode")
    return out


def prefill(pool: Pool, layer, slots, cu_seqlens, qkv, conv_w, g, beta, has_init=None):
    """Token-by-token prefill of N packed sequences; returns out [T][H][V]."""
    slots = _c(slots, np.int32)
    cu = _c(cu_seqlens, np.int32)
    N = slots.shape[0]
    T = int(cu[-1])
    qkv = _c(qkv, pool.io_np()).reshape(T, pool.D)
    g = _gate_arr(pool, g, (T,))
    beta = _c(beta, np.float32).reshape(T, pool.H)
    w = _c(conv_w, np.float32).reshape(pool.D, 4)
    hi = None if has_init is None else _c(has_init, np.uint8)
    out = np.zeros((T, pool.H, pool.V), pool.io_np())
    st = pool._struct()
    _check(_load().orc_prefill(ctypes.byref(st), layer, _ptr(slots), _ptr(cu), N, _ptr(hi),
                               _ptr(qkv), _ptr(w), _ptr(g), _ptr(beta), _ptr(out)), "prefill")
    return out


def slot_copy(pool: Pool, layer, src, dst, mask=None):
    src, dst = _c(src, np.int32), _c(dst, np.int32)
    m = None if mask is None else _c(mask, np.uint8)
    st = pool._struct()
    _check(_load().orc_slot_copy(ctypes.byref(st), layer, _ptr(src), _ptr(dst), _ptr(m),
                                 src.shape[0]), "slot_copy")


def spec_verify(pool: Pool, layer, slots, T, Lc, qkv, conv_w, g, beta):
    """Returns (spec_ssm [B][Lc][H][V][K], spec_conv [B][Lc][3][D], out [B][T][H][V]).
    Entries t >= T of the cache are left zero."""
    slots = _c(slots, np.int32)
    B = slots.shape[0]
    qkv = _c(qkv, pool.io_np()).reshape(B, T, pool.D)
    g = _gate_arr(pool, g, (B, T))
    beta = _c(beta, np.float32).reshape(B, T, pool.H)
    w = _c(conv_w, np.float32).reshape(pool.D, 4)
    spec_ssm = np.zeros((B, Lc, pool.H, pool.V, pool.K), storage_np_dtype(pool.state_dtype))
    spec_conv = np.zeros((B, Lc, 3, pool.D), pool.io_np())
    out = np.zeros((B, T, pool.H, pool.V), pool.io_np())
    st = pool._struct()
    _check(_load().orc_spec_verify(ctypes.byref(st), layer, _ptr(slots), B, T, Lc,
                                   _ptr(spec_ssm), _ptr(spec_conv), _ptr(qkv), _ptr(w),
                                   _ptr(g), _ptr(beta), _ptr(out)), "spec_verify")
    return spec_ssm, spec_conv, out


def spec_commit(pool: Pool, layer, slots, T, Lc, spec_ssm, spec_conv, accept):
    slots, acc = _c(slots, np.int32), _c(accept, np.int32)
    ss = _c(spec_ssm, storage_np_dtype(pool.state_dtype))
    sc = _c(spec_conv, pool.io_np())
    st = pool._struct()
    _check(_load().orc_spec_commit(ctypes.byref(st), layer, _ptr(slots), slots.shape[0], T,
                                   Lc, _ptr(ss), _ptr(sc), _ptr(acc)), "spec_commit")


def softplus(x: float) -> float:
    return _load().orc_softplus(float(x))


def sigmoid(x: float) -> float:
    return _load().orc_sigmoid(float(x))


def gates_from_raw(pool: "Pool", a, b, A_log, dt_bias):
    """(g, beta) of a batch from the raw projections (the gating reading of the C file)."""
    b = _c(b, np.float32)
    lead = b.shape[:-1]
    B = int(np.prod(lead)) if lead else 1
    n = pool.K if pool.gate == KDA else 1
    a = _c(a, np.float32).reshape(B, pool.H, n)
    A_log = _c(A_log, np.float32).reshape(pool.H)
    dt_bias = _c(dt_bias, np.float32).reshape(pool.H, n)
    g = np.empty((B, pool.H, n), np.float32)
    beta = np.empty((B, pool.H), np.float32)
    _load().orc_gates_from_raw(B, pool.H, pool.K, pool.gate, _ptr(a), _ptr(b.reshape(B, pool.H)),
                               _ptr(A_log), _ptr(dt_bias), _ptr(g), _ptr(beta))
    gshape = lead + ((pool.H, pool.K) if pool.gate == KDA else (pool.H,))
    return g.reshape(gshape), beta.reshape(lead + (pool.H,))


def decode_step_track(pool: "Pool", layer, slots, qkv, conv_w, g, beta, mask, track_slots):
    """Decode, then the masked track copy of the updated rows; returns out [B][H][V]."""
    slots, ts = _c(slots, np.int32), _c(track_slots, np.int32)
    mask = _c(mask, np.uint8)
    B = slots.shape[0]
    qkv = _c(qkv, pool.io_np()).reshape(B, pool.D)
    g = _gate_arr(pool, g, (B,))
    beta = _c(beta, np.float32).reshape(B, pool.H)
    w = _c(conv_w, np.float32).reshape(pool.D, 4)
    out = np.zeros((B, pool.H, pool.V), pool.io_np())
    st = pool._struct()
    _check(_load().orc_decode_step_track(ctypes.byref(st), layer, _ptr(slots), B, _ptr(qkv), _ptr(w),
                                         _ptr(g), _ptr(beta), _ptr(out), _ptr(mask), _ptr(ts)),
           "decode_step_track")
    return out


def decode_step_gated(pool: "Pool", layer, slots, qkv, conv_w, a, b, A_log, dt_bias):
    """Decode with the gates computed from raw projections; returns out [B][H][V]."""
    slots = _c(slots, np.int32)
    B = slots.shape[0]
    n = pool.K if pool.gate == KDA else 1
    qkv = _c(qkv, pool.io_np()).reshape(B, pool.D)
    w = _c(conv_w, np.float32).reshape(pool.D, 4)
    a = _c(a, np.float32).reshape(B, pool.H, n)
    b = _c(b, np.float32).reshape(B, pool.H)
    A_log = _c(A_log, np.float32).reshape(pool.H)
    dt_bias = _c(dt_bias, np.float32).reshape(pool.H, n)
    out = np.zeros((B, pool.H, pool.V), pool.io_np())
    st = pool._struct()
    _check(_load().orc_decode_step_gated(ctypes.byref(st), layer, _ptr(slots), B, _ptr(qkv), _ptr(w),
                                         _ptr(a), _ptr(b), _ptr(A_log), _ptr(dt_bias), _ptr(out)),
           "decode_step_gated")
    return out


class Rings:
    """ReplaySSM rings of a pool (numpy, mutated in place): per layer, pool row, head and
    entry: d [V], k [K], rawv [V], rawk [K] in the state dtype; g [K] (KDA) or [1] (GDN) and
    beta in fp32.  Shapes [layers][P+1][H][depth][n]."""

    def __init__(self, pool: "Pool", depth: int):
        L, R, H, K, V = pool.num_layers, pool.num_slots + 1, pool.H, pool.K, pool.V
        sd = storage_np_dtype(pool.state_dtype)
        gn = K if pool.gate == KDA else 1
        self.depth = depth
        self.d = np.zeros((L, R, H, depth, V), sd)
        self.k = np.zeros((L, R, H, depth, K), sd)
        self.rawv = np.zeros((L, R, H, depth, V), sd)
        self.rawk = np.zeros((L, R, H, depth, K), sd)
        self.g = np.zeros((L, R, H, depth, gn), np.float32)
        self.beta = np.zeros((L, R, H, depth), np.float32)

    def _struct(self):
        return _Rings(self.depth, _ptr(self.d), _ptr(self.k), _ptr(self.rawv), _ptr(self.rawk),
                      _ptr(self.g), _ptr(self.beta))


def replay_verify(pool: Pool, rings: Rings, layer, slots, pos, T, Lc, qkv, conv_w, g, beta):
    """ReplaySSM verify: records of token t go to ring entry (pos[b] + t) mod depth; the slot
    is not modified.  Returns (spec_conv [B][Lc][3][D], out [B][T][H][V])."""
    slots, pos = _c(slots, np.int32), _c(pos, np.int32)
    B = slots.shape[0]
    qkv = _c(qkv, pool.io_np()).reshape(B, T, pool.D)
    g = _gate_arr(pool, g, (B, T))
    beta = _c(beta, np.float32).reshape(B, T, pool.H)
    w = _c(conv_w, np.float32).reshape(pool.D, 4)
    spec_conv = np.zeros((B, Lc, 3, pool.D), pool.io_np())
    out = np.zeros((B, T, pool.H, pool.V), pool.io_np())
    st, rs = pool._struct(), rings._struct()
    _check(_load().orc_replay_verify(ctypes.byref(st), ctypes.byref(rs), layer, _ptr(slots),
                                     _ptr(pos), B, T, Lc, _ptr(spec_conv), _ptr(qkv), _ptr(w),
                                     _ptr(g), _ptr(beta), _ptr(out)), "replay_verify")
    return spec_conv, out


def replay_commit(pool: Pool, rings: Rings, layer, slots, pos, T, Lc, spec_conv, accept):
    """ReplaySSM commit: replay tokens 0..accept[b] from the slot state out of the rings,
    store the state into the slot and the window snapshot spec_conv[b][accept[b]]."""
    slots, pos, acc = _c(slots, np.int32), _c(pos, np.int32), _c(accept, np.int32)
    sc = _c(spec_conv, pool.io_np())
    st, rs = pool._struct(), rings._struct()
    _check(_load().orc_replay_commit(ctypes.byref(st), ctypes.byref(rs), layer, _ptr(slots),
                                     _ptr(pos), slots.shape[0], T, Lc, _ptr(sc), _ptr(acc)),
           "replay_commit")


# ----------------------------------------------------------------------------- pieces

def conv_sequence(win, x, w):
    """Short conv over T tokens from window win [3][D]; returns (new window, y [T][D])."""
    x = _c(x, np.float64)
    T, D = x.shape
    win = _c(win, np.float64).reshape(3, D).copy()
    w = _c(w, np.float32).reshape(D, 4)
    y = np.empty((T, D), np.float64)
    _load().orc_conv_sequence(D, T, _ptr(win), _ptr(x), _ptr(w), _ptr(y))
    return win, y


def recurrent_head(q, k, v, g, beta, S0):
    """Token-by-token gated delta rule of one head; returns (S_T, o [T][V], d [T][V])."""
    q, k, v = _c(q, np.float64), _c(k, np.float64), _c(v, np.float64)
    T, K = k.shape
    V = v.shape[1]
    g = _c(g, np.float64).reshape(T, K)
    beta = _c(beta, np.float64).reshape(T)
    S = _c(S0, np.float64).reshape(V, K).copy()
    o = np.empty((T, V), np.float64)
    d = np.empty((T, V), np.float64)
    _load().orc_recurrent_head(T, K, V, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                               _ptr(S), _ptr(o), _ptr(d))
    return S, o, d


def chunkwise_head(q, k, v, g, beta, S0, C=64):
    """Chunkwise WY/UT form of recurrent_head; returns (S_T, o [T][V])."""
    q, k, v = _c(q, np.float64), _c(k, np.float64), _c(v, np.float64)
    T, K = k.shape
    V = v.shape[1]
    g = _c(g, np.float64).reshape(T, K)
    beta = _c(beta, np.float64).reshape(T)
    S = _c(S0, np.float64).reshape(V, K).copy()
    o = np.empty((T, V), np.float64)
    _check(_load().orc_chunkwise_head(T, K, V, C, _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                      _ptr(beta), _ptr(S), _ptr(o)), "chunkwise")
    return S, o
