"""Seeded synthetic inputs shaped like the pages' workloads.

This module only draws random numbers and converts them to storage types; it holds
none of the layer step's arithmetic.  Both the CUDA path's tests/benchmark and the CPU
oracle take their inputs from here, so the two sides see identical bytes.

Distributions (workload statements of the hybrid-linear-attention cache pages; the
conv taps are not given there and are drawn N(0, 0.5)):
  q, k, v projections   N(0, 1)
  beta                  sigmoid(N(0, 1))
  log-decay gate g      -softplus(N(0, 1))     (alpha = exp(g) in (0, 1)); tests of strong
                        decay scale it, -s softplus(N(0, 1)) with s up to e^3
                        per key channel for KDA, one per head for GDN
  initial S, windows    N(0, 0.1)              (standard deviation 0.1)
  slot ids              distinct, uniform over the usable slots 1..P (row 0 is padding)
Storage arrays are numpy: fp32 as float32, bf16 as uint16 bit patterns (round to
nearest even from the float32 draw).
"""
from __future__ import annotations

import numpy as np

F32, BF16 = 0, 1
KDA, GDN = 0, 1


def rng(seed: int = 0) -> np.random.Generator:
    return np.random.default_rng(seed)


def f32_to_bf16_bits(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def storage(x, dt: int) -> np.ndarray:
    """float draw -> storage array of dtype dt (float32 or bf16 bits)."""
    x = np.asarray(x, np.float32)
    return x.copy() if dt == F32 else f32_to_bf16_bits(x)


def _sigmoid(z):
    return 1.0 / (1.0 + np.exp(-z))


def _neg_softplus(z):
    return -np.logaddexp(0.0, z)


def conv_weights(r: np.random.Generator, H: int, K: int, V: int, std: float = 0.5):
    D = H * (2 * K + V)
    return (r.standard_normal((D, 4)) * std).astype(np.float32)


def distinct_slots(r: np.random.Generator, B: int, P: int) -> np.ndarray:
    if B > P:
        raise ValueError("more requests than usable slots")
    return (r.permutation(P)[:B] + 1).astype(np.int32)


def gates(r: np.random.Generator, lead: tuple, H: int, K: int, gate: int, scale: float = 1.0):
    """(g, beta) for a leading shape (e.g. (B,), (T,), (B, T)).  scale multiplies the
    log-decay draw: g = -scale * softplus(N(0, 1)) (strong decay for scale >> 1)."""
    gshape = lead + ((H, K) if gate == KDA else (H,))
    g = (scale * _neg_softplus(r.standard_normal(gshape))).astype(np.float32)
    beta = _sigmoid(r.standard_normal(lead + (H,))).astype(np.float32)
    return g, beta


def projections(r: np.random.Generator, lead: tuple, H: int, K: int, V: int, io: int):
    D = H * (2 * K + V)
    return storage(r.standard_normal(lead + (D,)), io)


def pool_arrays(r: np.random.Generator, num_layers: int, num_slots: int, H: int, K: int,
                V: int, state_dtype: int, conv_dtype: int, std: float = 0.1):
    """(ssm [L][P+1][H][V][K], conv [L][P+1][3][D]) with every row ~ N(0, std)."""
    D = H * (2 * K + V)
    rows = num_slots + 1
    ssm = storage(r.standard_normal((num_layers, rows, H, V, K)) * std, state_dtype)
    conv = storage(r.standard_normal((num_layers, rows, 3, D)) * std, conv_dtype)
    return ssm, conv


def accept_counts(r: np.random.Generator, B: int, T: int) -> np.ndarray:
    """Accepted draft count per request, uniform over 0..T-1 (T = anchor + drafts)."""
    return r.integers(0, T, size=B).astype(np.int32)


def cu_seqlens(lengths) -> np.ndarray:
    return np.concatenate([[0], np.cumsum(np.asarray(lengths, np.int64))]).astype(np.int32)
