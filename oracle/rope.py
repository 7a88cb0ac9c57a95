"""Rotary position embedding, NeoX pairing -- TEST INFRASTRUCTURE ONLY (see
the package docstring for who may use it).

Follows "nx_f32_llama_v4b.nx source", Block section, RoPE step: each row's
position is its sequence's current length, a cos/sin table is built for that
position from head_dim and the base, and the "neox" application is made to
every query head and every new key head before the attend call.  The bodies
of the table builder and of the application are not printed on the pages;
this is the plain reading of the NeoX form:

    theta_i = base ** (-2 i / head_dim),     i = 0 .. head_dim/2 - 1
    angle   = pos * theta_i
    y[i]           = x[i] cos(angle) - x[i + head_dim/2] sin(angle)
    y[i + hd/2]    = x[i] sin(angle) + x[i + head_dim/2] cos(angle)

everything in float64.  V is not rotated.
"""
from __future__ import annotations

import numpy as np


def rope_neox(x, positions, head_dim: int, base: float) -> np.ndarray:
    """Rotate every head of every row of x.

    x: [T, n_heads * head_dim] (any float dtype; computed in float64);
    positions: [T] integer positions; returns float64 [T, n_heads*head_dim]."""
    x = np.asarray(x, dtype=np.float64)
    T, D = x.shape
    if head_dim % 2 != 0 or D % head_dim != 0:
        raise ValueError("head_dim must be even and divide the row width")
    half = head_dim // 2
    i = np.arange(half, dtype=np.float64)
    theta = float(base) ** (-2.0 * i / head_dim)                            # [half]
    ang = np.asarray(positions, dtype=np.float64)[:, None] * theta[None, :]  # [T, half]
    c, s = np.cos(ang), np.sin(ang)
    xh = x.reshape(T, D // head_dim, head_dim)
    a, b = xh[..., :half], xh[..., half:]
    y = np.empty_like(xh)
    y[..., :half] = a * c[:, None, :] - b * s[:, None, :]
    y[..., half:] = a * s[:, None, :] + b * c[:, None, :]
    return y.reshape(T, D)


def rope_neox_f32(x, positions, head_dim: int, base: float) -> np.ndarray:
    """The same rotation carried out in float32 the way the library's kernel
    does it -- cos and sin of the float64 angle rounded to float32, each
    product and each sum rounded to float32 -- for tests that must take the
    same rounding decision downstream (a bf16 pool rounds the rotated keys).
    Returns float32."""
    x = np.asarray(x, dtype=np.float32)
    T, D = x.shape
    if head_dim % 2 != 0 or D % head_dim != 0:
        raise ValueError("head_dim must be even and divide the row width")
    half = head_dim // 2
    i = np.arange(half, dtype=np.float64)
    theta = float(base) ** (-2.0 * i / head_dim)
    ang = np.asarray(positions, dtype=np.float64)[:, None] * theta[None, :]
    c = np.cos(ang).astype(np.float32)[:, None, :]
    s = np.sin(ang).astype(np.float32)[:, None, :]
    xh = x.reshape(T, D // head_dim, head_dim)
    a, b = xh[..., :half], xh[..., half:]
    y = np.empty_like(xh)
    y[..., :half] = (a * c) - (b * s)      # float32 operations, each rounded
    y[..., half:] = (a * s) + (b * c)
    return y.reshape(T, D)
