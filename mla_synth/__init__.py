"""Seeded synthetic inputs for one MLA decode step.

This module describes the five decode workloads (their shapes, dtypes and
seeds) and draws their random tensors. It holds none of the MLA arithmetic:
it only samples Gaussians, rounds them to the storage dtype and hands the same
values to both sides of every comparison (the fp64 oracle and the CUDA
library).

Recipe (applies to every workload):
  * one NumPy ``PCG64`` stream per tensor, spawned in a fixed order from
    ``SeedSequence(20261202 + workload_index)``;
  * hidden states ``h ~ N(0, 1)``; every weight ``W ~ N(0, 1/fan_in)`` where
    fan_in is the matrix's input width;
  * values are drawn in fp64 and rounded once, round-to-nearest-even, to the
    workload dtype (bf16 or fp32).
Long contexts (millions of tokens) are drawn on the GPU with a seeded
``torch.Generator`` per sequence instead (``context_h_device``), because the
host would need minutes; the oracle then receives copies of the sampled
sequences' rows.
"""
from __future__ import annotations

from dataclasses import dataclass, field
import numpy as np

__all__ = [
    "MLAShape", "WORKLOADS", "workload", "bf16_round", "bf16_bits", "bf16_bits_to_f64",
    "f32_round", "to_dtype", "draw_weights", "draw_new_tokens", "draw_context_lengths",
    "draw_context_h", "draw_latent_rows", "draw_absorbed_queries", "context_h_device",
    "WEIGHT_NAMES",
]

SEED_BASE = 20261202

# Order of the per-tensor streams (fixed; never reorder).
STREAM_ORDER = ("W_DKV", "W_KR", "W_DQ", "W_UQ", "W_QR", "W_UK", "W_UV", "W_O",
                "h_new", "ctx_len", "h_ctx", "rows", "q_abs", "spare0", "spare1")
WEIGHT_NAMES = STREAM_ORDER[:8]


@dataclass(frozen=True)
class MLAShape:
    """Dimensions of one MLA layer plus the decode batch that runs on it."""
    name: str
    index: int            # position in the workload list; selects the seed
    d: int                # hidden width
    n_h: int              # attention heads
    d_h: int              # per-head content (and value) width
    d_c: int              # KV latent width (cached)
    d_r: int              # decoupled RoPE width (cached, shared by all heads)
    d_cq: int             # query latent width (not cached)
    batch: int
    ctx: int              # cached tokens per sequence before the new one (0 = ragged)
    ragged_max: int = 0   # ragged: context ~ Uniform[1, ragged_max]
    dtype: str = "bf16"   # "bf16" or "f32"
    rope_base: float = 10000.0
    note: str = ""

    @property
    def D(self) -> int:
        """Width of one cache row: latent c_KV followed by the RoPE key k_R."""
        return self.d_c + self.d_r

    @property
    def seed(self) -> int:
        return SEED_BASE + self.index

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == "bf16" else 4

    def fan_in(self, name: str) -> int:
        return {"W_DKV": self.d, "W_KR": self.d, "W_DQ": self.d,
                "W_UQ": self.d_cq, "W_QR": self.d_cq,
                "W_UK": self.d_c, "W_UV": self.d_c,
                "W_O": self.n_h * self.d_h}[name]

    def weight_shape(self, name: str) -> tuple[int, int]:
        """Row-major [out, in] storage, as nn.Linear keeps it."""
        return {"W_DKV": (self.d_c, self.d), "W_KR": (self.d_r, self.d),
                "W_DQ": (self.d_cq, self.d),
                "W_UQ": (self.n_h * self.d_h, self.d_cq),
                "W_QR": (self.n_h * self.d_r, self.d_cq),
                "W_UK": (self.n_h * self.d_h, self.d_c),
                "W_UV": (self.n_h * self.d_h, self.d_c),
                "W_O": (self.d, self.n_h * self.d_h)}[name]

    def scaled(self, **kw) -> "MLAShape":
        """Same layer with a different batch / context (for small parity cases)."""
        d = dict(self.__dict__)
        d.update(kw)
        return MLAShape(**d)


WORKLOADS = {
    "tiny": MLAShape("tiny", 0, d=256, n_h=4, d_h=32, d_c=64, d_r=16, d_cq=96,
                     batch=2, ctx=128, dtype="f32",
                     note="tiny MLA decode, fp32, batch 2, context 128"),
    "minimind": MLAShape("minimind", 1, d=768, n_h=8, d_h=96, d_c=128, d_r=32, d_cq=256,
                         batch=256, ctx=2048, dtype="bf16",
                         note="MiniMind-shaped small-head MLA decode, bf16, batch 256, context 2048"),
    "v2": MLAShape("v2", 2, d=5120, n_h=128, d_h=128, d_c=512, d_r=64, d_cq=1536,
                   batch=64, ctx=4096, dtype="bf16",
                   note="DeepSeek-V2-shaped MLA decode, bf16, batch 64, context 4096"),
    "v2_ragged": MLAShape("v2_ragged", 3, d=5120, n_h=128, d_h=128, d_c=512, d_r=64, d_cq=1536,
                          batch=128, ctx=0, ragged_max=32768, dtype="bf16",
                          note="V2 shape, bf16, batch 128, context ~ Uniform[1, 32768]"),
    "v2_long": MLAShape("v2_long", 4, d=5120, n_h=128, d_h=128, d_c=512, d_r=64, d_cq=1536,
                        batch=8, ctx=131072, dtype="bf16",
                        note="V2 shape, bf16, batch 8, context 131072"),
}


def workload(name: str) -> MLAShape:
    return WORKLOADS[name]


# --------------------------------------------------------------------------
# rounding of drawn values to the storage dtype
# --------------------------------------------------------------------------
def bf16_round(x) -> np.ndarray:
    """Round fp64 values once, to nearest-even, onto the bf16 grid (result fp64)."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                 # x = m * 2**e, 0.5 <= |m| < 1
    r = np.rint(m * 256.0) / 256.0     # 8 significant bits; rint is ties-to-even
    return np.ldexp(r, e)


def f32_round(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def bf16_bits(x) -> np.ndarray:
    """uint16 bit patterns of values that already lie on the bf16 grid."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32)
    if np.any(u & 0xFFFF):
        raise ValueError("bf16_bits: value not on the bf16 grid")
    return (u >> 16).astype(np.uint16)


def bf16_bits_to_f64(bits) -> np.ndarray:
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def to_dtype(x, dtype: str) -> np.ndarray:
    return bf16_round(x) if dtype == "bf16" else f32_round(x)


# --------------------------------------------------------------------------
# streams
# --------------------------------------------------------------------------
def _stream(shape: MLAShape, name: str, sub: int | None = None) -> np.random.Generator:
    ss = np.random.SeedSequence(shape.seed).spawn(len(STREAM_ORDER))[STREAM_ORDER.index(name)]
    if sub is not None:
        ss = np.random.SeedSequence(entropy=ss.entropy, spawn_key=ss.spawn_key + (sub,))
    return np.random.Generator(np.random.PCG64(ss))


def draw_weights(shape: MLAShape) -> dict[str, np.ndarray]:
    """All eight projection matrices, fp64 arrays holding dtype-rounded values."""
    out = {}
    for name in WEIGHT_NAMES:
        rows, cols = shape.weight_shape(name)
        w = _stream(shape, name).standard_normal((rows, cols)) * np.sqrt(1.0 / shape.fan_in(name))
        out[name] = to_dtype(w, shape.dtype)
    return out


def draw_new_tokens(shape: MLAShape, batch: int | None = None) -> np.ndarray:
    """Hidden states of the token being decoded, one per sequence: [B, d]."""
    B = shape.batch if batch is None else batch
    return to_dtype(_stream(shape, "h_new").standard_normal((B, shape.d)), shape.dtype)


def draw_context_lengths(shape: MLAShape, batch: int | None = None) -> np.ndarray:
    """Cached tokens per sequence before the new one (the new token sits at this position)."""
    B = shape.batch if batch is None else batch
    if shape.ctx > 0:
        return np.full(B, shape.ctx, dtype=np.int64)
    return _stream(shape, "ctx_len").integers(1, shape.ragged_max, endpoint=True, size=B)


def draw_context_h(shape: MLAShape, b: int, n_tokens: int) -> np.ndarray:
    """Hidden states of sequence b's cached tokens (host; for small contexts): [n, d]."""
    g = _stream(shape, "h_ctx", sub=b)
    return to_dtype(g.standard_normal((n_tokens, shape.d)), shape.dtype)


def context_h_device(shape: MLAShape, b: int, n_tokens: int, device, start: int = 0):
    """Hidden states of sequence b's cached tokens drawn on the GPU: bf16 [n, d].

    Deterministic in (seed, b): rows [start, start+n) of one per-sequence draw,
    generated chunk by chunk (each chunk of 8192 tokens has its own seed), so a
    sampled sequence can be regenerated or copied to the host for the oracle.
    """
    import torch
    CH = 8192
    outs = []
    t = start
    end = start + n_tokens
    while t < end:
        c = t // CH
        lo = c * CH
        g = torch.Generator(device=device)
        g.manual_seed(shape.seed * 1_000_003 + b * 65_537 + c)
        blk = torch.randn((CH, shape.d), generator=g, device=device, dtype=torch.float32)
        a, z = t - lo, min(end, lo + CH) - lo
        outs.append(blk[a:z].to(torch.bfloat16 if shape.dtype == "bf16" else torch.float32))
        t = lo + z
    return torch.cat(outs, 0) if outs else torch.empty((0, shape.d), device=device)


def draw_gaussian(shape: MLAShape, tag: str, dims, sub: int = 0, std: float = 1.0) -> np.ndarray:
    """A stand-alone tensor of the workload dtype, every element ~ N(0, std^2),
    from its own seeded stream (tag, sub)."""
    g = _stream(shape, tag, sub=sub)
    return to_dtype(g.standard_normal(tuple(dims)) * std, shape.dtype)


def draw_latent_rows(shape: MLAShape, n_rows: int, sub: int = 0) -> np.ndarray:
    """Stand-alone cache rows [n, d_c + d_r] with the statistics the append path
    produces under this recipe (every element ~ N(0, 1))."""
    g = _stream(shape, "rows", sub=sub)
    return to_dtype(g.standard_normal((n_rows, shape.D)), shape.dtype)


def draw_absorbed_queries(shape: MLAShape, batch: int, sub: int = 0) -> np.ndarray:
    """Stand-alone absorbed queries [B, n_h, d_c + d_r]: the latent part has the
    variance d_h/d_c that W_UK^T q_C has under this recipe, the RoPE part unit
    variance, so scaled scores have unit variance (near-uniform attention)."""
    g = _stream(shape, "q_abs", sub=sub)
    q = g.standard_normal((batch, shape.n_h, shape.D))
    q[..., :shape.d_c] *= np.sqrt(shape.d_h / shape.d_c)
    return to_dtype(q, shape.dtype)
