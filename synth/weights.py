"""Seeded random decoder weights.

Every linear and embedding matrix is drawn as ``standard_normal * 0.02`` in
fp32, in one fixed tensor order:

    embed; for each layer: q, k, v, o, gate, up, down; lm_head (untied only)

Matrices use the ``[out_features][in_features]`` layout.  Norm gains are 1
(the N(0, 0.02) law applies to linear and embedding matrices only).  For the
bf16 shapes each fp32 draw is rounded to the nearest bf16 (ties to even) and
kept as its 16-bit pattern.

Tensor ``i`` of the order is drawn in chunks of ``CHUNK`` elements; chunk
``j`` uses its own PCG64 stream seeded by ``SeedSequence(seed,
spawn_key=(i, j))``.  The values therefore do not depend on how many threads
fill them, and the chunks fill in parallel (numpy releases the GIL in bulk
draws and ufuncs).
"""
from __future__ import annotations

import os
import struct
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np

from .shapes import ModelConfig

CHUNK = 1 << 22
STD = 0.02


@dataclass
class Weights:
    cfg: ModelConfig
    embed: np.ndarray                      # [V][d]
    layers: List[dict] = field(default_factory=list)
    final_norm: Optional[np.ndarray] = None  # [d] fp32
    lm_head: Optional[np.ndarray] = None     # [V][d] or None when tied

    @property
    def is_bf16(self) -> bool:
        return self.embed.dtype == np.uint16

    def matrices(self):
        """(name, array) for every matrix, in the fixed draw order."""
        yield "embed", self.embed
        for i, lw in enumerate(self.layers):
            for k in ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down"):
                yield f"layers.{i}.{k}", lw[k]
        if self.lm_head is not None:
            yield "lm_head", self.lm_head


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Reinterpret bf16 bit patterns as the fp32 numbers they denote (exact)."""
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def _round_to_bf16_bits(x: np.ndarray, out: np.ndarray) -> None:
    """fp32 -> bf16 bit pattern, round to nearest, ties to even (finite input)."""
    u = x.view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    u += np.uint32(0x7FFF)
    u += lsb
    np.right_shift(u, np.uint32(16), out=u)
    out[...] = u


def _fill_tensor(shape, tensor_index: int, seed: int, as_bf16: bool, pool) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16 if as_bf16 else np.float32)
    n_chunks = (n + CHUNK - 1) // CHUNK

    def work(j: int) -> None:
        lo, hi = j * CHUNK, min(n, (j + 1) * CHUNK)
        ss = np.random.SeedSequence(seed, spawn_key=(tensor_index, j))
        g = np.random.Generator(np.random.PCG64(ss))
        buf = g.standard_normal(hi - lo, dtype=np.float32)
        buf *= np.float32(STD)
        if as_bf16:
            _round_to_bf16_bits(buf, out[lo:hi])
        else:
            out[lo:hi] = buf

    list(pool.map(work, range(n_chunks)))
    return out.reshape(shape)


def make_weights(cfg: ModelConfig, seed: int = 0, threads: Optional[int] = None) -> Weights:
    """Draw the decoder's weights (see module docstring for the recipe)."""
    as_bf16 = cfg.dtype == "bf16"
    d, F, V = cfg.d_model, cfg.d_ff, cfg.vocab
    threads = threads or min(32, os.cpu_count() or 1)
    idx = 0
    with ThreadPoolExecutor(max_workers=threads) as pool:
        def nxt(shape):
            nonlocal idx
            t = _fill_tensor(shape, idx, seed, as_bf16, pool)
            idx += 1
            return t

        embed = nxt((V, d))
        layers = []
        for _ in range(cfg.n_layers):
            lw = {
                "wq": nxt((cfg.q_dim, d)),
                "wk": nxt((cfg.kv_dim, d)),
                "wv": nxt((cfg.kv_dim, d)),
                "wo": nxt((d, cfg.q_dim)),
                "w_gate": nxt((F, d)),
                "w_up": nxt((F, d)),
                "w_down": nxt((d, F)),
                "attn_norm": np.ones(d, dtype=np.float32),
                "mlp_norm": np.ones(d, dtype=np.float32),
            }
            layers.append(lw)
        lm_head = None if cfg.tied_embedding else nxt((V, d))
    return Weights(cfg, embed, layers, np.ones(d, dtype=np.float32), lm_head)


# ---------------------------------------------------------------------------
# .pcdw file: a 64-byte header, then every tensor in a fixed order.
#   header: b"PCDW", u32 version=1, u32 dtype (1 = f32, 2 = bf16),
#           u32 n_layers, d_model, n_q_heads, n_kv_heads, head_dim, d_ff,
#           vocab, tied, reserved(0), f32 rms_eps, f32 rope_theta,
#           zero padding to 64 B.
#   body:   embed; per layer: attn_norm(f32), wq, wk, wv, wo, mlp_norm(f32),
#           w_gate, w_up, w_down; final_norm(f32); lm_head (untied only).
#   Matrices are stored in the header's dtype, norm gains always as f32.
# ---------------------------------------------------------------------------
PCDW_MAGIC = b"PCDW"


def write_pcdw(w: Weights, path: str) -> None:
    c = w.cfg
    hdr = PCDW_MAGIC + struct.pack(
        "<11I2f", 1, 2 if w.is_bf16 else 1, c.n_layers, c.d_model, c.n_q_heads,
        c.n_kv_heads, c.head_dim, c.d_ff, c.vocab, 1 if c.tied_embedding else 0, 0,
        c.rms_eps, c.rope_theta)
    hdr = hdr.ljust(64, b"\0")
    with open(path, "wb") as f:
        f.write(hdr)
        f.write(np.ascontiguousarray(w.embed).tobytes())
        for lw in w.layers:
            f.write(lw["attn_norm"].astype(np.float32).tobytes())
            for k in ("wq", "wk", "wv", "wo"):
                f.write(np.ascontiguousarray(lw[k]).tobytes())
            f.write(lw["mlp_norm"].astype(np.float32).tobytes())
            for k in ("w_gate", "w_up", "w_down"):
                f.write(np.ascontiguousarray(lw[k]).tobytes())
        f.write(w.final_norm.astype(np.float32).tobytes())
        if w.lm_head is not None:
            f.write(np.ascontiguousarray(w.lm_head).tobytes())
