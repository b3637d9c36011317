"""Shared helpers for the GPU parity tests: moving generator values to the
device, building a decoder, and the tolerance checks."""
from __future__ import annotations

import numpy as np

import mla_synth as S

# Tolerances. bf16 storage with fp32 accumulation: max|err| <= 1e-2 * max|ref| and
# per-row relative L2 <= 5e-3 (rows: one (sequence, head) of o_lat / q_abs, one
# sequence of u, one cache row). fp32 storage: both bounds at 2e-5.
TOL = {"bf16": (1e-2, 5e-3), "f32": (2e-5, 2e-5)}
# The whole step chains six stored bf16 roundings (cache, c_Q, q_C, q_abs,
# o_lat, o) before u. Each adds about 1.6e-3 relative RMS error (uniform
# rounding on the bf16 grid) and the attention weights inherit the score error
# (about 3e-3 relative on o_lat); the root-sum-square is about 5e-3, so the
# per-row bound doubles the single-stage one.
TOL_E2E = {"bf16": (2e-2, 1.2e-2), "f32": (5e-5, 5e-5)}
# Absolute LSE error of the whole step. The LSE moves by the softmax-weighted
# mean of the score errors, so it is bounded by the largest one. A score is a
# dot product of two stored vectors; each bf16 rounding of a stored operand
# (cache row, c_Q, q_C, q_abs: four stages) perturbs a unit-variance score by
# about 2^-9/sqrt(3) = 1.1e-3 RMS, 2.3e-3 together; 1e-2 is over four of those
# standard deviations even when one row takes all the weight. fp32 storage
# leaves only accumulation-order error.
TOL_LSE_E2E = {"bf16": 1e-2, "f32": 1e-4}
# The same bound for checks over ~10^5 LSE values (many query rows, each with
# its own score errors; a query that sees only itself has the error of one
# score): the largest of n Gaussian errors reaches sqrt(2 ln n) = 4.8 standard
# deviations of 2.3e-3 at n = 10^5, so the bound is 6.5 of them.
TOL_LSE_E2E_MANY = {"bf16": 1.5e-2, "f32": 1e-4}


def torch_dtype(shape):
    import torch
    return torch.bfloat16 if shape.dtype == "bf16" else torch.float32


def dev(x, shape, dtype=None):
    """Host fp64 array (already on the dtype grid) -> CUDA tensor of the workload dtype."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(np.asarray(x, dtype=np.float64)))
    return t.to(dtype or torch_dtype(shape)).cuda().contiguous()


def dev_i32(x):
    import torch
    return torch.as_tensor(np.asarray(x, dtype=np.int32)).cuda().contiguous()


def host(t):
    import torch
    return t.detach().to(torch.float64).cpu().numpy()


def errors(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    err = got - ref
    max_rel = np.abs(err).max() / max(np.abs(ref).max(), 1e-300)
    r2 = ref.reshape(-1, ref.shape[-1])
    e2 = err.reshape(-1, ref.shape[-1])
    rn = np.linalg.norm(r2, axis=1)
    nz = rn > 0
    row = (np.linalg.norm(e2[nz], axis=1) / rn[nz]).max() if nz.any() else 0.0
    assert np.all(e2[~nz] == 0), "rows whose reference is zero must be exactly zero"
    return max_rel, row


def assert_close(got, ref, dtype, tol=None, what=""):
    tmax, trow = (tol or TOL)[dtype]
    max_rel, row = errors(got, ref)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    assert max_rel <= tmax and row <= trow, f"{what}: max|d|/max|ref| = {max_rel:.3e} (<= {tmax}), " \
                                            f"row rel L2 = {row:.3e} (<= {trow})"
    return max_rel, row


def make_weights_dev(shape, W):
    return {k: dev(v, shape) for k, v in W.items()}


def decoder(shape, W_dev, batch, max_len, max_pos=None):
    import head_latent_attention_24_b300 as M
    ls = M.LayerShape(shape.d, shape.n_h, shape.d_h, shape.d_c, shape.d_r, shape.d_cq, shape.dtype, shape.rope_base)
    return M.MLADecoder(ls, W_dev, batch, max_len, max_pos=max_pos)
