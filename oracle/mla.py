"""Plain fp64 CPU oracle for one decode step of Multi-head Latent Attention (MLA).

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports this module:
only ``tests/``, the smoke check in ``__graft_entry__`` and the benchmark's
CPU-baseline leg use it. It shares no code with the CUDA library.

Every function is the plain definition from the pages, in fp64 NumPy, with
library matmuls as the only building block. No blocking, fusion or reordering.

Pages cited (title, then section):
  [Latent]   "Latent 压缩"                                   (zdszero.github.io/latent.html)
  [MLA]      "MLA：潜在表示压缩与解耦 RoPE"                     (lizn-zn.github.io, scholia-log)
  [MiniMind] "MiniMind 学习笔记 10：Multi-Latent Attention，从 KV Cache
              压缩到 MiniMind 改造思路"                          (p-chao.com)

Conventions: weights are stored row-major [out, in] as nn.Linear keeps them
([MiniMind] §9) and act on column vectors ([MLA] §3). Head i owns rows
[i*d_h, (i+1)*d_h) of W_UQ, W_UK and W_UV, rows [i*d_r, (i+1)*d_r) of W_QR and
columns [i*d_h, (i+1)*d_h) of W_O ([MLA] §4, the per-head form of u_t).

Readings where the pages leave a step open: RoPE is the rotate-half form with inverse frequencies
base^(-2j/d_r), j < d_r/2 — the pages never define RoPE, and [MiniMind] §6/§9
apply it through ``apply_rotary_pos_emb(q, k, cos, sin)`` on the rope slice
only (§12 sizes the table by the rope width). The decode query attends to every
cached row including its own ([MiniMind] §12, causal mask with cache). The
latent is cached as projected ([MLA] has no norm); the variant that applies
[MiniMind] §9's kv_norm (an RMSNorm over the kv_lora_rank latent before it is
cached) takes its weight and epsilon as arguments (the pages give neither
value).

Pins: every function here is checked in tests/test_oracle_pins.py against
something other than itself (closed forms, the pages' printed numbers, brute
force on tiny inputs, library routines). None is "parity unpinned".
"""
from __future__ import annotations

import numpy as np

F64 = np.float64


def _f64(x):
    return np.asarray(x, dtype=F64)


def per_token_cache_elems(d_c: int, d_r: int) -> int:
    """Elements cached per token per layer: the latent c_KV plus the shared RoPE
    key k_R ([MLA] §6 last paragraph; §8 prints 512 + 64 = 576)."""
    return d_c + d_r


def scale_of(d_h: int, d_r: int) -> float:
    """Softmax temperature 1/sqrt(d_h + d_r) ([MLA] §7, a = softmax(q^T k / sqrt(d_h+d_r)))."""
    return 1.0 / np.sqrt(float(d_h + d_r))


# --------------------------------------------------------------------------
# RoPE (reading: rotate-half form; see module docstring)
# --------------------------------------------------------------------------
def rope_inv_freq(d_r: int, base: float) -> np.ndarray:
    """theta_j = base^(-2j/d_r) for j < d_r/2 ([MiniMind] §12: table over the rope width)."""
    j = np.arange(d_r // 2, dtype=F64)
    return np.power(F64(base), -2.0 * j / d_r)


def rope(x, pos, base: float) -> np.ndarray:
    """Rotate the last axis of x (width d_r) by position pos.

    Pair (x_j, x_{j+d_r/2}) is turned by the angle pos * theta_j:
        y_j          = x_j cos - x_{j+d_r/2} sin
        y_{j+d_r/2}  = x_{j+d_r/2} cos + x_j sin
    ``pos`` broadcasts against x[..., 0].
    """
    x = _f64(x)
    d_r = x.shape[-1]
    half = d_r // 2
    ang = _f64(pos)[..., None] * rope_inv_freq(d_r, base)
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


# --------------------------------------------------------------------------
# Step S1: what one token writes into the latent cache
# --------------------------------------------------------------------------
def rms_norm(x, weight, eps: float) -> np.ndarray:
    """RMSNorm over the last axis: x / sqrt(mean(x^2) + eps) * weight
    ([MiniMind] §9: ``self.kv_norm = RMSNorm(self.kv_lora_rank, eps=...)``,
    applied as ``kv_latent = self.kv_norm(kv_latent)``)."""
    x = _f64(x)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + F64(eps)) * _f64(weight)


def cache_rows(h, W_DKV, W_KR, pos, base: float, kv_norm_weight=None, kv_norm_eps: float = 1e-5) -> np.ndarray:
    """Cache rows [c_KV ‖ k_R] for tokens h [N, d] at positions pos [N].

    c_KV = W_DKV h           ([MLA] §3 down-projection; [Latent] "MLA：latent 作为可缓存的 KV 表示")
    k_R  = RoPE(W_KR h)      ([MLA] §6, shared by all heads, computed from h directly)
    Row layout: latent first, then the rope key ([MiniMind] §9: kv_down_proj
    output split as [kv_lora_rank, qk_rope_head_dim], cache = (kv_latent, k_rope)).
    With kv_norm_weight given, the latent is RMS-normalised before it is cached
    ([MiniMind] §9, the kv_norm variant); the rope key is not.
    """
    h = _f64(h)
    c_kv = h @ _f64(W_DKV).T
    if kv_norm_weight is not None:
        c_kv = rms_norm(c_kv, kv_norm_weight, kv_norm_eps)
    k_r = rope(h @ _f64(W_KR).T, pos, base)
    return np.concatenate([c_kv, k_r], axis=-1)


# --------------------------------------------------------------------------
# Step S2: the query, absorbed into latent space
# --------------------------------------------------------------------------
def absorbed_query(h, W_DQ, W_UQ, W_QR, W_UK, pos, n_h: int, d_h: int, d_r: int,
                   base: float, return_parts: bool = False):
    """q_abs [B, n_h, d_c + d_r] = [q~_i ‖ q_R_i] for new tokens h [B, d] at pos [B].

    c_Q  = W_DQ h                      ([MLA] §3, query low-rank path)
    q_C  = W_UQ c_Q   (per head i)     ([MLA] §3; §7 full forward)
    q_R  = RoPE(W_QR c_Q) per head     ([MLA] §6, one rope query per head)
    q~_i = W_UK_i^T q_C_i              ([MLA] §4 matrix absorption;
                                        [Latent] <q, W_K c> = <W_K^T q, c>)
    """
    h = _f64(h)
    B = h.shape[0]
    W_UK = _f64(W_UK)
    d_c = W_UK.shape[1]
    c_q = h @ _f64(W_DQ).T
    q_c = (c_q @ _f64(W_UQ).T).reshape(B, n_h, d_h)
    q_r = rope((c_q @ _f64(W_QR).T).reshape(B, n_h, d_r), _f64(pos)[:, None], base)
    W_UK_heads = W_UK.reshape(n_h, d_h, d_c)
    q_tilde = np.einsum("bik,ikc->bic", q_c, W_UK_heads)
    q_abs = np.concatenate([q_tilde, q_r], axis=-1)
    if return_parts:
        return q_abs, {"c_Q": c_q, "q_C": q_c, "q_R": q_r, "q_tilde": q_tilde}
    return q_abs


# --------------------------------------------------------------------------
# Step S3: attention in latent space
# --------------------------------------------------------------------------
def latent_attention(q_abs, rows, d_c: int, scale: float):
    """One sequence: q_abs [n_h, d_c + d_r], cache rows [L, d_c + d_r].

    score_{i,t} = (q~_i^T c_KV_t + q_R_i^T k_R_t) * scale   ([MLA] §6 two-part score, §7 scale)
    a_{i,t}     = softmax over t                            ([MLA] §7)
    o_lat_i     = sum_t a_{i,t} c_KV_t                      ([MLA] §4 u_t formula, inner sum;
                                                             [Latent] value deferral)
    lse_i       = log sum_t exp(score_{i,t})  (natural log, scaled scores)
    Two-pass softmax (max, then exponentials). L = 0 gives o_lat = 0, lse = -inf.
    """
    q_abs = _f64(q_abs)
    rows = _f64(rows)
    n_h = q_abs.shape[0]
    if rows.shape[0] == 0:
        return np.zeros((n_h, d_c)), np.full(n_h, -np.inf)
    s = (q_abs @ rows.T) * scale
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    l = e.sum(axis=1, keepdims=True)
    o_lat = (e @ rows[:, :d_c]) / l
    lse = (m + np.log(l))[:, 0]
    return o_lat, lse


# --------------------------------------------------------------------------
# Steps S4/S5: expand by W_UV_i, then W_O
# --------------------------------------------------------------------------
def output_projection(o_lat, W_UV, W_O, n_h: int, d_h: int, return_o: bool = False):
    """u = sum_i W_O_i W_UV_i o_lat_i for o_lat [B, n_h, d_c]  ([MLA] §4, u_t formula; §7 u = W_O o)."""
    o_lat = _f64(o_lat)
    B, _, d_c = o_lat.shape
    W_UV_heads = _f64(W_UV).reshape(n_h, d_h, d_c)
    o = np.einsum("bic,ikc->bik", o_lat, W_UV_heads).reshape(B, n_h * d_h)
    u = o @ _f64(W_O).T
    return (u, o) if return_o else u


# --------------------------------------------------------------------------
# The pre-merged weight forms ([MLA] §4)
# --------------------------------------------------------------------------
def premerged_query_weights(W_UQ, W_UK, n_h: int, d_h: int):
    """W_QK [n_h, d_c, d_cq] with W_QK_i = W_UK_i^T W_UQ_i.

    [MLA] §4: W^{UQ T} W^{UK} can be merged ahead of time, so the content
    score is c_Q^T (W_UQ_i^T W_UK_i) c_KV. Stored as the map that takes c_Q
    straight to q~_i = W_QK_i c_Q.
    """
    W_UQ = _f64(W_UQ)
    W_UK = _f64(W_UK)
    d_cq, d_c = W_UQ.shape[1], W_UK.shape[1]
    UQ = W_UQ.reshape(n_h, d_h, d_cq)
    UK = W_UK.reshape(n_h, d_h, d_c)
    return np.stack([UK[i].T @ UQ[i] for i in range(n_h)])


def premerged_output_weights(W_UV, W_O, n_h: int, d_h: int):
    """W_OUV [d, n_h * d_c] whose column block i is W_O_i W_UV_i.

    [MLA] §4, the per-head u_t formula u = sum_i W_O_i W_UV_i o_lat_i: with the
    product merged ahead of time u = W_OUV [o_lat_1; ...; o_lat_nh].
    """
    W_UV = _f64(W_UV)
    W_O = _f64(W_O)
    d_c = W_UV.shape[1]
    UV = W_UV.reshape(n_h, d_h, d_c)
    return np.concatenate([W_O[:, i * d_h:(i + 1) * d_h] @ UV[i] for i in range(n_h)], axis=1)


# --------------------------------------------------------------------------
# The whole step, two ways
# --------------------------------------------------------------------------
def decode_absorbed(h_ctx_list, h_new, W, n_h, d_h, d_r, base, pos=None, kv_norm_weight=None,
                    kv_norm_eps: float = 1e-5):
    """The four steps chained (append every token, absorbed query, latent
    attention over rows 0..pos, output projection). Returns (u, o_lat, lse, q_abs, rows).
    kv_norm_weight: the [MiniMind] §9 variant that RMS-normalises the cached latent."""
    h_new = _f64(h_new)
    B = h_new.shape[0]
    d_c = W["W_DKV"].shape[0]
    if pos is None:
        pos = np.array([len(hc) for hc in h_ctx_list])
    scale = scale_of(d_h, d_r)
    q_abs = absorbed_query(h_new, W["W_DQ"], W["W_UQ"], W["W_QR"], W["W_UK"], pos, n_h, d_h, d_r, base)
    o_lat = np.zeros((B, n_h, d_c))
    lse = np.zeros((B, n_h))
    rows_all = []
    for b in range(B):
        L = int(pos[b])
        toks = np.concatenate([_f64(h_ctx_list[b])[:L], h_new[b:b + 1]], axis=0)
        rows = cache_rows(toks, W["W_DKV"], W["W_KR"], np.arange(L + 1), base, kv_norm_weight, kv_norm_eps)
        rows_all.append(rows)
        o_lat[b], lse[b] = latent_attention(q_abs[b], rows, d_c, scale)
    u = output_projection(o_lat, W["W_UV"], W["W_O"], n_h, d_h)
    return u, o_lat, lse, q_abs, rows_all


def decode_materialised(h_ctx_list, h_new, W, n_h, d_h, d_r, base, pos=None, return_parts=False,
                        kv_norm_weight=None, kv_norm_eps: float = 1e-5):
    """The decode step as plain multi-head attention over materialised K and V.

    For every cached token (positions 0..pos-1) and the new token (position pos):
      c_KV = W_DKV h, k_R = RoPE(W_KR h)                            ([MLA] §3, §6)
      per head i: k_C = W_UK_i c_KV, v_C = W_UV_i c_KV, k = [k_C ; k_R]  ([MLA] §7;
                  [MiniMind] §10 naive version: K_nope, V restored, k_rope expanded to all heads)
    New token: c_Q = W_DQ h, q_C = W_UQ_i c_Q, q_R = RoPE(W_QR_i c_Q), q = [q_C ; q_R]
    a = softmax(q^T k / sqrt(d_h + d_r)) over all rows 0..pos   ([MLA] §7; [MiniMind] §12)
    o_i = sum_t a_t v_C,t ; u = W_O [o_1; ...; o_nh]            ([MLA] §7)
    Nothing is absorbed here: this is the definition the absorbed path must reach.
    With kv_norm_weight, c_KV is RMS-normalised before K and V are expanded from it
    ([MiniMind] §9: kv_latent = kv_norm(kv_latent), then kv_up_proj).
    Returns u [B, d] (and per-sequence o [B, n_h*d_h], lse [B, n_h] if asked).
    """
    h_new = _f64(h_new)
    B, d = h_new.shape
    W = {k: _f64(v) for k, v in W.items()}
    d_c = W["W_DKV"].shape[0]
    if pos is None:
        pos = np.array([len(hc) for hc in h_ctx_list])
    scale = scale_of(d_h, d_r)
    u = np.zeros((B, d))
    o_all = np.zeros((B, n_h * d_h))
    lse_all = np.zeros((B, n_h))
    for b in range(B):
        L = int(pos[b])
        toks = np.concatenate([_f64(h_ctx_list[b])[:L], h_new[b:b + 1]], axis=0)   # [L+1, d]
        c_kv = toks @ W["W_DKV"].T                                                     # [L+1, d_c]
        if kv_norm_weight is not None:
            c_kv = rms_norm(c_kv, kv_norm_weight, kv_norm_eps)
        k_r = rope(toks @ W["W_KR"].T, np.arange(L + 1), base)                         # [L+1, d_r]
        # k_C = W_UK c_KV and v_C = W_UV c_KV for every row, all heads stacked ([MLA] §3)
        k_c = (c_kv @ W["W_UK"].T).reshape(L + 1, n_h, d_h).transpose(1, 0, 2)        # [n_h, L+1, d_h]
        v_c = (c_kv @ W["W_UV"].T).reshape(L + 1, n_h, d_h).transpose(1, 0, 2)        # [n_h, L+1, d_h]
        k = np.concatenate([k_c, np.broadcast_to(k_r, (n_h,) + k_r.shape)], axis=-1)   # [n_h, L+1, d_h+d_r]
        c_q = h_new[b] @ W["W_DQ"].T
        q_c = (W["W_UQ"] @ c_q).reshape(n_h, d_h)
        q_r = rope((W["W_QR"] @ c_q).reshape(n_h, d_r), np.full(n_h, float(L)), base)
        q = np.concatenate([q_c, q_r], axis=-1)                                        # [n_h, d_h+d_r]
        s = np.matmul(k, q[:, :, None])[:, :, 0] * scale                              # [n_h, L+1]
        m = s.max(axis=1, keepdims=True)
        e = np.exp(s - m)
        l = e.sum(axis=1, keepdims=True)
        a = e / l
        o = np.matmul(a[:, None, :], v_c)[:, 0, :]                                     # [n_h, d_h]
        o_all[b] = o.reshape(-1)
        lse_all[b] = (m + np.log(l))[:, 0]
        u[b] = W["W_O"] @ o.reshape(-1)
    if return_parts:
        return u, o_all, lse_all
    return u


# --------------------------------------------------------------------------
# The materialised (MHA) path for several query tokens per sequence
# --------------------------------------------------------------------------
def materialised_kv(rows, W_UK, W_UV, n_h: int, d_h: int):
    """k_C [N, n_h, d_h] = W_UK_i c_KV and v_C [N, n_h, d_h] = W_UV_i c_KV for
    cache rows [N, d_c + d_r] ([MLA] §3 low-rank K/V; [MiniMind] §10 naive
    version: K_nope and V restored from the latent)."""
    rows = _f64(rows)
    d_c = _f64(W_UK).shape[1]
    c_kv = rows[:, :d_c]
    N = rows.shape[0]
    k_c = (c_kv @ _f64(W_UK).T).reshape(N, n_h, d_h)
    v_c = (c_kv @ _f64(W_UV).T).reshape(N, n_h, d_h)
    return k_c, v_c


def materialised_query(h, W_DQ, W_UQ, W_QR, pos, n_h: int, d_h: int, d_r: int, base: float):
    """q [N, n_h, d_h + d_r] = [W_UQ_i c_Q ; RoPE(W_QR_i c_Q)], c_Q = W_DQ h
    ([MLA] §3 and §6), for tokens h [N, d] at positions pos [N]."""
    h = _f64(h)
    N = h.shape[0]
    c_q = h @ _f64(W_DQ).T
    q_c = (c_q @ _f64(W_UQ).T).reshape(N, n_h, d_h)
    q_r = rope((c_q @ _f64(W_QR).T).reshape(N, n_h, d_r), _f64(pos)[:, None], base)
    return np.concatenate([q_c, q_r], axis=-1)


def mha_attention(q, k_c, k_r, v_c, q_pos, scale: float):
    """Causal multi-head attention of one sequence over materialised keys.

    q [T, n_h, d_h + d_r] at positions q_pos [T]; k_c [L, n_h, d_h], the shared
    RoPE key k_r [L, d_r] and v_c [L, n_h, d_h] of rows 0..L-1. Query t sees
    rows 0..q_pos[t] ([MiniMind] §12: with a cache the query sees every earlier
    row and itself); k = [k_C ; k_R] per head ([MLA] §6), scale 1/sqrt(d_h+d_r)
    ([MLA] §7). Two-pass softmax. Returns o [T, n_h, d_h] and the natural-log
    LSE [T, n_h].
    """
    q, k_c, k_r, v_c = _f64(q), _f64(k_c), _f64(k_r), _f64(v_c)
    T, n_h, _ = q.shape
    L = k_c.shape[0]
    k = np.concatenate([k_c, np.broadcast_to(k_r[:, None, :], (L, n_h, k_r.shape[1]))], axis=-1)
    s = np.einsum("thc,lhc->htl", q, k) * scale                          # [n_h, T, L]
    visible = np.arange(L)[None, :] <= _f64(q_pos)[:, None]               # [T, L]
    s = np.where(visible[None], s, -np.inf)
    m = s.max(axis=2, keepdims=True)
    e = np.exp(s - m)
    l = e.sum(axis=2, keepdims=True)
    o = np.einsum("htl,lhc->thc", e / l, v_c)
    lse = (m + np.log(l))[:, :, 0].T
    return o, lse


def prefill_materialised(h_ctx_list, h_new_list, W, n_h, d_h, d_r, base, return_parts=False):
    """Several new tokens per sequence through the materialised (MHA) path.

    [Latent]: at prefill MLA takes the MHA path (K and V restored from the
    latent); [MiniMind] §10 naive version. Sequence b holds L_b cached tokens
    h_ctx_list[b] at positions 0..L_b-1 and T_b new tokens h_new_list[b] at
    positions L_b..L_b+T_b-1; every new token is appended to the cache and
    then attends causally. Returns u per sequence [T_b, d] (and o [T_b, n_h*d_h],
    lse [T_b, n_h] per sequence if asked).
    """
    W = {k: _f64(v) for k, v in W.items()}
    scale = scale_of(d_h, d_r)
    us, os_, lses = [], [], []
    for h_ctx, h_new in zip(h_ctx_list, h_new_list):
        h_ctx, h_new = _f64(h_ctx), _f64(h_new)
        L, T = h_ctx.shape[0], h_new.shape[0]
        toks = np.concatenate([h_ctx, h_new], axis=0)
        rows = cache_rows(toks, W["W_DKV"], W["W_KR"], np.arange(L + T), base)
        k_c, v_c = materialised_kv(rows, W["W_UK"], W["W_UV"], n_h, d_h)
        q_pos = L + np.arange(T)
        q = materialised_query(h_new, W["W_DQ"], W["W_UQ"], W["W_QR"], q_pos, n_h, d_h, d_r, base)
        d_c = W["W_DKV"].shape[0]
        o, lse = mha_attention(q, k_c, rows[:, d_c:], v_c, q_pos, scale)
        o = o.reshape(T, n_h * d_h)
        us.append(o @ W["W_O"].T)
        os_.append(o)
        lses.append(lse)
    return (us, os_, lses) if return_parts else us
