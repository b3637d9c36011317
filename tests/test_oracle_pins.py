"""Pins for the fp64 oracle: each check ties an oracle function to something
other than itself — the pages' printed numbers, closed forms, brute force on
tiny inputs, or a library routine. A second group plants plausible mistakes in
copies of the oracle's functions and shows that a pin catches each one.

CPU only (no GPU marker).
"""
import json
import math
import os

import numpy as np
import pytest
from scipy.special import logsumexp

import oracle
from oracle import mla as O
import mla_synth as S

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_numbers.json")


def golden():
    with open(GOLDEN) as f:
        return json.load(f)


# A micro layer small enough for pure-Python loops.
MICRO = dict(d=8, n_h=2, d_h=4, d_c=4, d_r=2, d_cq=6)


def micro_inputs(seed=7, L=3, scale_w=1.0):
    rng = np.random.default_rng(seed)
    m = MICRO
    W = {
        "W_DKV": rng.standard_normal((m["d_c"], m["d"])) * scale_w,
        "W_KR": rng.standard_normal((m["d_r"], m["d"])) * scale_w,
        "W_DQ": rng.standard_normal((m["d_cq"], m["d"])) * scale_w,
        "W_UQ": rng.standard_normal((m["n_h"] * m["d_h"], m["d_cq"])) * scale_w,
        "W_QR": rng.standard_normal((m["n_h"] * m["d_r"], m["d_cq"])) * scale_w,
        "W_UK": rng.standard_normal((m["n_h"] * m["d_h"], m["d_c"])) * scale_w,
        "W_UV": rng.standard_normal((m["n_h"] * m["d_h"], m["d_c"])) * scale_w,
        "W_O": rng.standard_normal((m["d"], m["n_h"] * m["d_h"])) * scale_w,
    }
    h_ctx = [rng.standard_normal((L, m["d"])) * 0.3]
    h_new = rng.standard_normal((1, m["d"])) * 0.3
    return W, h_ctx, h_new


# ---------------------------------------------------------------------------
# brute force: plain Python loops, written from the definitions, no numpy math
# ---------------------------------------------------------------------------
def _matvec(Wm, x):
    return [sum(float(Wm[r][c]) * float(x[c]) for c in range(len(x))) for r in range(len(Wm))]


def _rope_complex(x, p, base):
    """RoPE written through complex numbers: pair j is the complex number
    x_j + i x_{j+d/2}, multiplied by e^{i p theta_j}, theta_j = exp(-(2j/d) ln base)."""
    d = len(x)
    half = d // 2
    out = [0.0] * d
    for j in range(half):
        theta = math.exp(-(2.0 * j / d) * math.log(base))
        z = complex(x[j], x[j + half]) * complex(math.cos(p * theta), math.sin(p * theta))
        out[j], out[j + half] = z.real, z.imag
    return out


def brute_force_mha(W, h_ctx, h_new, n_h, d_h, d_r, base):
    """Standard multi-head attention over explicitly built K and V, loops only."""
    d_c = len(W["W_DKV"])
    toks = [list(r) for r in h_ctx] + [list(h_new)]
    L1 = len(toks)
    pos_new = L1 - 1
    keys, vals = [], []
    for t, x in enumerate(toks):
        c = _matvec(W["W_DKV"], x)
        kr = _rope_complex(_matvec(W["W_KR"], x), t, base)
        kc = _matvec(W["W_UK"], c)       # all heads stacked
        vc = _matvec(W["W_UV"], c)
        keys.append([kc[i * d_h:(i + 1) * d_h] + kr for i in range(n_h)])
        vals.append([vc[i * d_h:(i + 1) * d_h] for i in range(n_h)])
    cq = _matvec(W["W_DQ"], h_new)
    qc = _matvec(W["W_UQ"], cq)
    qr_all = _matvec(W["W_QR"], cq)
    o = []
    for i in range(n_h):
        q = qc[i * d_h:(i + 1) * d_h] + _rope_complex(qr_all[i * d_r:(i + 1) * d_r], pos_new, base)
        s = [sum(q[k] * keys[t][i][k] for k in range(d_h + d_r)) / math.sqrt(d_h + d_r) for t in range(L1)]
        mx = max(s)
        e = [math.exp(v - mx) for v in s]
        tot = sum(e)
        o += [sum(e[t] / tot * vals[t][i][k] for t in range(L1)) for k in range(d_h)]
    return _matvec(W["W_O"], o)


# ---------------------------------------------------------------------------
# pins: the pages' printed numbers
# ---------------------------------------------------------------------------
def test_cache_size_numbers_v2():
    g = golden()
    dims = g["v2_dims"]["values"]
    per_tok = O.per_token_cache_elems(dims["d_c"], dims["d_r"])
    mha = 2 * dims["n_h"] * dims["d_h"]
    assert per_tok == g["v2_mla_cache_per_token"]["value"]
    assert mha == g["v2_mha_cache_per_token"]["value"]
    assert round(100.0 * per_tok / mha, g["v2_ratio_percent"]["digits"]) == g["v2_ratio_percent"]["value"]
    assert round(mha / per_tok) == g["v2_ratio_fold"]["value"]
    assert per_tok / (2 * dims["d_h"]) == g["v2_gqa_equivalent_groups"]["value"]
    # the oracle's own cache row has exactly that width
    shp = S.workload("v2")
    assert (shp.d, shp.n_h, shp.d_h, shp.d_c, shp.d_cq, shp.d_r) == tuple(
        dims[k] for k in ("d", "n_h", "d_h", "d_c", "d_cq", "d_r"))
    rng = np.random.default_rng(0)
    rows = O.cache_rows(rng.standard_normal((3, 16)), rng.standard_normal((dims["d_c"], 16)),
                        rng.standard_normal((dims["d_r"], 16)), np.arange(3), 10000.0)
    assert rows.shape == (3, 576)


def test_cache_size_numbers_minimind():
    g = golden()
    gqa = g["minimind_gqa_cache_per_token"]["values_from"]
    mla = g["minimind_mla_cache_per_token"]["values_from"]
    gqa_elems = gqa["num_key_value_heads"] * gqa["head_dim"] * 2
    mla_elems = O.per_token_cache_elems(mla["kv_lora_rank"], mla["qk_rope_head_dim"])
    assert gqa_elems == g["minimind_gqa_cache_per_token"]["value"]
    assert mla_elems == g["minimind_mla_cache_per_token"]["value"]
    assert round(100 * mla_elems / gqa_elems, 1) == g["minimind_ratio_percent"]["value"]
    assert round(100 * (1 - mla_elems / gqa_elems), 1) == g["minimind_saving_percent"]["value"]
    shp = S.workload("minimind")
    assert shp.d_c + shp.d_r == mla_elems


# ---------------------------------------------------------------------------
# pins: RoPE
# ---------------------------------------------------------------------------
def check_rope_identity_at_zero(rope):
    x = np.random.default_rng(1).standard_normal((5, 16))
    return np.array_equal(rope(x, np.zeros(5), 10000.0), x)


def check_rope_closed_form_d2(rope):
    # d_r = 2: theta_0 = 1, so (1, 0) at position p turns into (cos p, sin p).
    ok = True
    for p in (0.0, 1.0, 2.5, 100.0, 131072.0):
        y = rope(np.array([[1.0, 0.0]]), np.array([p]), 10000.0)[0]
        ok &= abs(y[0] - math.cos(p)) < 1e-12 and abs(y[1] - math.sin(p)) < 1e-12
    return ok


def check_rope_complex(rope, base=10000.0):
    rng = np.random.default_rng(2)
    ok = True
    for d in (2, 16, 32, 64):
        for p in (0, 1, 17, 4096, 131072):
            x = rng.standard_normal(d)
            ok &= np.allclose(rope(x[None], np.array([p]), base)[0], _rope_complex(list(x), p, base),
                              rtol=0, atol=1e-9)
    return ok


def check_rope_relative(rope, base=10000.0):
    # <R_t q, R_s k> depends on s - t only (MLA page §5: R_t^T R_s = R_{s-t}).
    rng = np.random.default_rng(3)
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    ok = True
    for t, s, delta in ((5, 9, 100), (0, 4096, 7), (4096, 0, 131000), (3, 3, 12345)):
        a = rope(q[None], np.array([t]), base)[0] @ rope(k[None], np.array([s]), base)[0]
        b = rope(q[None], np.array([t + delta]), base)[0] @ rope(k[None], np.array([s + delta]), base)[0]
        c = q @ rope(k[None], np.array([s - t]), base)[0]
        ok &= abs(a - b) < 1e-8 * (1 + abs(a)) and abs(a - c) < 1e-8 * (1 + abs(a))
    return ok


def test_rope_pins():
    assert check_rope_identity_at_zero(O.rope)
    assert check_rope_closed_form_d2(O.rope)
    assert check_rope_complex(O.rope)
    assert check_rope_relative(O.rope)
    x = np.random.default_rng(4).standard_normal((9, 32))
    y = O.rope(x, np.arange(9) * 1000, 10000.0)
    assert np.allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-13)


def test_rope_inv_freq_values():
    f = O.rope_inv_freq(64, 10000.0)
    assert f.shape == (32,)
    assert f[0] == 1.0
    assert abs(f[16] - 0.01) < 1e-15          # 10000^(-32/64) = 1/100
    assert abs(f[31] - 10000.0 ** (-62 / 64)) < 1e-18


# ---------------------------------------------------------------------------
# pins: append (S1)
# ---------------------------------------------------------------------------
def check_cache_rows_unit_vectors(cache_rows):
    rng = np.random.default_rng(5)
    Wd, Wr = rng.standard_normal((8, 12)), rng.standard_normal((4, 12))
    ok = True
    for k in range(12):
        e = np.zeros((1, 12))
        e[0, k] = 1.0
        r = cache_rows(e, Wd, Wr, np.array([0]), 10000.0)[0]
        ok &= np.array_equal(r, np.concatenate([Wd[:, k], Wr[:, k]]))
    # a position other than 0 only turns the rope part
    e = np.zeros((1, 12))
    e[0, 3] = 1.0
    r = cache_rows(e, Wd, Wr, np.array([37]), 10000.0)[0]
    ok &= np.array_equal(r[:8], Wd[:, 3])
    ok &= np.allclose(r[8:], _rope_complex(list(Wr[:, 3]), 37, 10000.0), atol=1e-12)
    return ok


def test_cache_rows_unit_vectors():
    assert check_cache_rows_unit_vectors(O.cache_rows)


def test_key_rank_bound():
    # rank(W_UK W_DKV) <= d_c, and the materialised keys of many tokens span at
    # most d_c directions (Latent page: rank(W_eff) <= L; MLA page §3).
    rng = np.random.default_rng(6)
    n_h, d_h, d_c, d = 8, 16, 24, 96
    W_UK, W_DKV = rng.standard_normal((n_h * d_h, d_c)), rng.standard_normal((d_c, d))
    sv = np.linalg.svd(W_UK @ W_DKV, compute_uv=False)
    assert sv[d_c - 1] > 1e-6 * sv[0]
    assert np.all(sv[d_c:] <= 1e-10 * sv[0])
    h = rng.standard_normal((200, d))
    rows = O.cache_rows(h, W_DKV, rng.standard_normal((4, d)), np.arange(200), 10000.0)
    K = rows[:, :d_c] @ W_UK.T          # [tokens, n_h*d_h]
    sk = np.linalg.svd(K, compute_uv=False)
    assert np.all(sk[d_c:] <= 1e-10 * sk[0])


# ---------------------------------------------------------------------------
# pins: absorption (S2) and latent attention (S3)
# ---------------------------------------------------------------------------
def check_absorption_identity(absorbed_query, cache_rows):
    """q^T k (materialised, per head) equals q_abs . row (absorbed) — MLA page §4/§6;
    and the content part equals c_Q^T (W_UQ_i^T W_UK_i) c_KV (pre-merged form, §4)."""
    m = MICRO
    W, h_ctx, h_new = micro_inputs(11, L=5)
    pos = np.array([5])
    q_abs = absorbed_query(h_new, W["W_DQ"], W["W_UQ"], W["W_QR"], W["W_UK"], pos,
                           m["n_h"], m["d_h"], m["d_r"], 10000.0)[0]
    toks = np.concatenate([h_ctx[0], h_new])
    rows = cache_rows(toks, W["W_DKV"], W["W_KR"], np.arange(6), 10000.0)
    ok = True
    c_q = _matvec(W["W_DQ"], h_new[0])
    for i in range(m["n_h"]):
        WUQ_i = W["W_UQ"][i * m["d_h"]:(i + 1) * m["d_h"]]
        WUK_i = W["W_UK"][i * m["d_h"]:(i + 1) * m["d_h"]]
        merged = WUQ_i.T @ WUK_i                     # d_cq x d_c
        q_c = WUQ_i @ np.array(c_q)
        q_r = _rope_complex(_matvec(W["W_QR"][i * m["d_r"]:(i + 1) * m["d_r"]], c_q), 5, 10000.0)
        for t in range(6):
            c_kv = rows[t, :m["d_c"]]
            k_c = WUK_i @ c_kv
            mat = q_c @ k_c + np.dot(q_r, rows[t, m["d_c"]:])
            pre = np.array(c_q) @ merged @ c_kv + np.dot(q_r, rows[t, m["d_c"]:])
            ab = q_abs[i] @ rows[t]
            ok &= abs(mat - ab) <= 1e-12 * (1 + abs(mat)) and abs(pre - ab) <= 1e-12 * (1 + abs(pre))
    return ok


def test_absorption_identity():
    assert check_absorption_identity(O.absorbed_query, O.cache_rows)


def test_value_deferral_identity():
    # sum_s a_s W_V c_s = W_V sum_s a_s c_s (Latent page), on the oracle's o_lat.
    rng = np.random.default_rng(12)
    n_h, d_c, d_r, L, d_h = 3, 10, 4, 17, 5
    q = rng.standard_normal((n_h, d_c + d_r))
    rows = rng.standard_normal((L, d_c + d_r))
    W_V = rng.standard_normal((d_h, d_c))
    o_lat, _ = O.latent_attention(q, rows, d_c, 0.3)
    s = 0.3 * q @ rows.T
    a = np.exp(s - s.max(1, keepdims=True))
    a /= a.sum(1, keepdims=True)
    lhs = np.stack([sum(a[i, t] * (W_V @ rows[t, :d_c]) for t in range(L)) for i in range(n_h)])
    assert np.allclose(lhs, o_lat @ W_V.T, rtol=1e-12, atol=1e-12)


def check_latent_attention_brute(latent_attention):
    rng = np.random.default_rng(13)
    ok = True
    for (n_h, d_c, d_r, L) in ((1, 2, 2, 1), (2, 3, 2, 4), (3, 4, 2, 7)):
        q = rng.standard_normal((n_h, d_c + d_r))
        rows = rng.standard_normal((L, d_c + d_r))
        sc = 0.7
        o, lse = latent_attention(q, rows, d_c, sc)
        for i in range(n_h):
            s = [sc * sum(q[i, k] * rows[t, k] for k in range(d_c + d_r)) for t in range(L)]
            ref_lse = logsumexp(s)
            w = [math.exp(v - ref_lse) for v in s]
            ref_o = [sum(w[t] * rows[t, c] for t in range(L)) for c in range(d_c)]
            ok &= abs(lse[i] - ref_lse) < 1e-12 and np.allclose(o[i], ref_o, rtol=1e-12, atol=1e-14)
    return ok


def check_latent_special_cases(latent_attention):
    rng = np.random.default_rng(14)
    d_c, d_r, n_h = 6, 2, 3
    ok = True
    # seqlen 1: the only row's latent, lse = its score
    q, r = rng.standard_normal((n_h, 8)), rng.standard_normal((1, 8))
    o, lse = latent_attention(q, r, d_c, 0.5)
    ok &= np.allclose(o, np.broadcast_to(r[0, :d_c], (n_h, d_c)), rtol=0, atol=1e-15)
    ok &= np.allclose(lse, 0.5 * q @ r[0], rtol=1e-14)
    # all rows equal: output is that row whatever the scores
    rows = np.tile(rng.standard_normal((1, 8)), (9, 1))
    o, lse = latent_attention(q, rows, d_c, 0.5)
    ok &= np.allclose(o, np.broadcast_to(rows[0, :d_c], (n_h, d_c)), atol=1e-14)
    ok &= np.allclose(lse, 0.5 * q @ rows[0] + math.log(9), rtol=1e-13)
    # q = 0: uniform weights, mean of the rows, lse = log L
    rows = rng.standard_normal((11, 8))
    o, lse = latent_attention(np.zeros((n_h, 8)), rows, d_c, 0.5)
    ok &= np.allclose(o, np.broadcast_to(rows[:, :d_c].mean(0), (n_h, d_c)), atol=1e-14)
    ok &= np.allclose(lse, math.log(11), rtol=1e-14)
    # empty: zeros and -inf
    o, lse = latent_attention(q, np.zeros((0, 8)), d_c, 0.5)
    ok &= np.all(o == 0) and np.all(np.isneginf(lse))
    return ok


def test_latent_attention_brute_force():
    assert check_latent_attention_brute(O.latent_attention)


def test_latent_attention_special_cases():
    assert check_latent_special_cases(O.latent_attention)


def test_latent_attention_rope_zeroed_is_mqa():
    # With the rope part zeroed the score is a plain MQA over the latent (Latent page:
    # decode is formally MQA with one latent head).
    rng = np.random.default_rng(15)
    q = rng.standard_normal((4, 10))
    q[:, 8:] = 0.0
    rows = rng.standard_normal((13, 10))
    o, lse = O.latent_attention(q, rows, 8, 0.25)
    s = 0.25 * q[:, :8] @ rows[:, :8].T
    assert np.allclose(lse, logsumexp(s, axis=1), rtol=1e-14)


# ---------------------------------------------------------------------------
# pins: whole step, both formulations against brute force
# ---------------------------------------------------------------------------
def check_materialised_vs_brute(decode_materialised, seed=21):
    m = MICRO
    W, h_ctx, h_new = micro_inputs(seed, L=4)
    u = decode_materialised(h_ctx, h_new, W, m["n_h"], m["d_h"], m["d_r"], 10000.0)[0]
    ref = brute_force_mha({k: v.tolist() for k, v in W.items()}, h_ctx[0].tolist(), h_new[0].tolist(),
                          m["n_h"], m["d_h"], m["d_r"], 10000.0)
    return np.allclose(u, ref, rtol=1e-11, atol=1e-12)


def test_materialised_vs_brute_force():
    assert check_materialised_vs_brute(O.decode_materialised)
    assert check_materialised_vs_brute(O.decode_materialised, seed=22)


def test_absorbed_equals_materialised_on_workload_shapes():
    # The absorbed chain (what the CUDA library computes) equals the materialised
    # definition on the tiny workload and on a MiniMind-shaped layer with a short context.
    for name, ctx in (("tiny", 128), ("minimind", 40)):
        shp = S.workload(name).scaled(batch=2, ctx=ctx)
        W = S.draw_weights(shp)
        h_new = S.draw_new_tokens(shp, 2)
        h_ctx = [S.draw_context_h(shp, b, ctx) for b in range(2)]
        u_m = O.decode_materialised(h_ctx, h_new, W, shp.n_h, shp.d_h, shp.d_r, shp.rope_base)
        u_a, o_lat, lse, q_abs, rows = O.decode_absorbed(h_ctx, h_new, W, shp.n_h, shp.d_h, shp.d_r,
                                                         shp.rope_base)
        assert np.allclose(u_a, u_m, rtol=1e-10, atol=1e-10 * np.abs(u_m).max())
        assert rows[0].shape == (ctx + 1, shp.D)
        # seqlen 1 special case of the whole step: u = W_O [W_UV_i c_KV_0]
    shp = S.workload("tiny").scaled(batch=1, ctx=0)
    W = S.draw_weights(shp)
    h_new = S.draw_new_tokens(shp, 1)
    u = O.decode_materialised([np.zeros((0, shp.d))], h_new, W, shp.n_h, shp.d_h, shp.d_r, shp.rope_base)
    c_kv = W["W_DKV"] @ h_new[0]
    o = np.concatenate([W["W_UV"][i * shp.d_h:(i + 1) * shp.d_h] @ c_kv for i in range(shp.n_h)])
    assert np.allclose(u[0], W["W_O"] @ o, rtol=1e-12, atol=1e-12)


def test_scale():
    assert O.scale_of(128, 64) == 1 / math.sqrt(192)
    assert O.scale_of(96, 32) == 1 / math.sqrt(128)


# ---------------------------------------------------------------------------
# planted mistakes: each mutant of an oracle function must fail a pin
# ---------------------------------------------------------------------------
def _rope_sign_flip(x, pos, base):
    y = O.rope(x, -np.asarray(pos, dtype=float), base)
    return y


def _rope_interleaved(x, pos, base):
    # pairs (x_{2j}, x_{2j+1}) instead of rotate-half
    x = np.asarray(x, float)
    d = x.shape[-1]
    perm = np.concatenate([np.arange(0, d, 2), np.arange(1, d, 2)])
    inv = np.argsort(perm)
    return O.rope(x[..., perm], pos, base)[..., inv]


def _rope_wrong_freq(x, pos, base):
    x = np.asarray(x, float)
    d = x.shape[-1]
    half = d // 2
    ang = np.asarray(pos, float)[..., None] * np.power(base, -np.arange(half) / d)
    c, s = np.cos(ang), np.sin(ang)
    return np.concatenate([x[..., :half] * c - x[..., half:] * s, x[..., half:] * c + x[..., :half] * s], -1)


def _cache_rows_swapped(h, W_DKV, W_KR, pos, base):
    r = O.cache_rows(h, W_DKV, W_KR, pos, base)
    d_r = W_KR.shape[0]
    return np.concatenate([r[:, -d_r:], r[:, :-d_r]], axis=1)


def _absorbed_wrong_head_layout(h, W_DQ, W_UQ, W_QR, W_UK, pos, n_h, d_h, d_r, base):
    # takes head i's rows of W_UK with a head-minor stride (rows k*n_h + i)
    q, parts = O.absorbed_query(h, W_DQ, W_UQ, W_QR, W_UK, pos, n_h, d_h, d_r, base, return_parts=True)
    d_c = np.asarray(W_UK).shape[1]
    Wt = np.asarray(W_UK).reshape(d_h, n_h, d_c).transpose(1, 0, 2)
    qt = np.einsum("bik,ikc->bic", parts["q_C"], Wt)
    return np.concatenate([qt, parts["q_R"]], -1)


def _absorbed_no_rope(h, W_DQ, W_UQ, W_QR, W_UK, pos, n_h, d_h, d_r, base):
    return O.absorbed_query(h, W_DQ, W_UQ, W_QR, W_UK, np.zeros_like(np.asarray(pos)), n_h, d_h, d_r, base)


def _latent_no_max(q, rows, d_c, scale):
    o, lse = O.latent_attention(q, rows, d_c, scale)
    return o, lse - np.log(max(1, np.asarray(rows).shape[0]))


def _latent_unnormalised(q, rows, d_c, scale):
    o, lse = O.latent_attention(q, rows, d_c, scale)
    return o * np.asarray(rows).shape[0] if np.asarray(rows).shape[0] else o, lse


def _latent_dropped_rope_term(q, rows, d_c, scale):
    q = np.array(q, float)
    q[:, d_c:] = 0
    return O.latent_attention(q, rows, d_c, scale)


def _materialised_scale(h_ctx, h_new, W, n_h, d_h, d_r, base):
    # 1/sqrt(d_h) instead of 1/sqrt(d_h + d_r): emulate by rescaling the query weights
    W2 = dict(W)
    f = math.sqrt((d_h + d_r) / d_h)
    W2["W_DQ"] = np.asarray(W["W_DQ"]) * f
    return O.decode_materialised(h_ctx, h_new, W2, n_h, d_h, d_r, base)


@pytest.mark.parametrize("mutant", [_rope_sign_flip, _rope_interleaved, _rope_wrong_freq])
def test_planted_rope_mistakes_are_caught(mutant):
    caught = not (check_rope_identity_at_zero(mutant) and check_rope_closed_form_d2(mutant)
                  and check_rope_complex(mutant) and check_rope_relative(mutant))
    assert caught


def test_planted_cache_row_mistake_is_caught():
    assert not check_cache_rows_unit_vectors(_cache_rows_swapped)


@pytest.mark.parametrize("mutant", [_absorbed_wrong_head_layout, _absorbed_no_rope])
def test_planted_absorption_mistakes_are_caught(mutant):
    assert not check_absorption_identity(mutant, O.cache_rows)


@pytest.mark.parametrize("mutant", [_latent_no_max, _latent_unnormalised, _latent_dropped_rope_term])
def test_planted_attention_mistakes_are_caught(mutant):
    assert not (check_latent_attention_brute(mutant) and check_latent_special_cases(mutant))


def test_planted_scale_mistake_is_caught():
    assert not check_materialised_vs_brute(_materialised_scale)


# ---------------------------------------------------------------------------
# pins: the kv_norm variant of S1 (MiniMind page §9: RMSNorm on the cached latent)
# ---------------------------------------------------------------------------
def check_rms_norm(fn):
    rng = np.random.default_rng(21)
    x = rng.standard_normal((6, 40)) * rng.uniform(0.1, 30.0, size=(6, 1))
    ones = np.ones(40)
    y = fn(x, ones, 0.0)
    ok = np.allclose(np.mean(y * y, axis=-1), 1.0, atol=1e-12)               # unit RMS
    ok &= np.allclose(np.abs(np.sum(y * x, -1)), np.linalg.norm(y, axis=-1) * np.linalg.norm(x, axis=-1),
                      rtol=1e-12)                                              # parallel to x
    ok &= bool(np.all(np.sum(y * x, -1) > 0))                                 # same direction
    ok &= np.allclose(fn(7.5 * x, ones, 0.0), y, atol=1e-12)                  # scale invariant
    w = rng.standard_normal(40)
    ok &= np.allclose(fn(x, w, 0.0), y * w, atol=1e-12)                       # weight is elementwise
    ok &= bool(np.all(fn(np.zeros((2, 40)), ones, 1e-5) == 0.0))              # zero row stays zero
    return bool(ok)


def test_rms_norm_pins():
    assert check_rms_norm(O.rms_norm)


def test_rms_norm_matches_library_routine():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(22)
    x, w = rng.standard_normal((5, 128)), rng.standard_normal(128)
    for eps in (1e-5, 1e-2):
        ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (128,), torch.from_numpy(w), eps).numpy()
        assert np.allclose(O.rms_norm(x, w, eps), ref, rtol=1e-12, atol=1e-14)


def check_cache_rows_kv_norm(cache_rows):
    rng = np.random.default_rng(23)
    d, d_c, d_r = 32, 16, 8
    h = rng.standard_normal((9, d))
    Wd, Wr = rng.standard_normal((d_c, d)), rng.standard_normal((d_r, d))
    pos = np.arange(9) * 5
    plain = cache_rows(h, Wd, Wr, pos, 10000.0)
    normed = cache_rows(h, Wd, Wr, pos, 10000.0, np.ones(d_c), 0.0)
    lat, lat0 = normed[:, :d_c], plain[:, :d_c]
    ok = np.allclose(np.mean(lat * lat, -1), 1.0, atol=1e-12)
    ok &= np.allclose(lat * np.sqrt(np.mean(lat0 * lat0, -1, keepdims=True)), lat0, atol=1e-12)
    ok &= np.array_equal(normed[:, d_c:], plain[:, d_c:])                    # the rope key is not normalised
    return bool(ok)


def test_cache_rows_kv_norm_pins():
    assert check_cache_rows_kv_norm(O.cache_rows)


def test_kv_norm_absorbed_equals_materialised():
    # With the latent normalised before caching, the absorbed chain (latent
    # cache, absorbed query, value deferral) still equals the materialised
    # definition (K and V expanded from the normalised latent).
    shp = S.workload("tiny")
    W = S.draw_weights(shp)
    rng = np.random.default_rng(24)
    g = rng.uniform(0.5, 1.5, size=shp.d_c)
    h_ctx = [S.draw_context_h(shp, b, n) for b, n in enumerate([40, 17])]
    h_new = S.draw_new_tokens(shp, 2)
    u_m = O.decode_materialised(h_ctx, h_new, W, shp.n_h, shp.d_h, shp.d_r, shp.rope_base, kv_norm_weight=g,
                                kv_norm_eps=1e-6)
    u_a = O.decode_absorbed(h_ctx, h_new, W, shp.n_h, shp.d_h, shp.d_r, shp.rope_base, kv_norm_weight=g,
                            kv_norm_eps=1e-6)[0]
    u_plain = O.decode_materialised(h_ctx, h_new, W, shp.n_h, shp.d_h, shp.d_r, shp.rope_base)
    assert np.allclose(u_a, u_m, rtol=1e-10, atol=1e-12)
    assert not np.allclose(u_m, u_plain, rtol=1e-3)                           # the norm changes the step


def _rms_norm_sum_not_mean(x, weight, eps):
    x = np.asarray(x, float)
    return x / np.sqrt(np.sum(x * x, -1, keepdims=True) + eps) * weight


def _rms_norm_eps_outside(x, weight, eps):
    x = np.asarray(x, float)
    return x / (np.sqrt(np.mean(x * x, -1, keepdims=True)) + 1e-3 + eps) * weight


def _cache_rows_norm_whole_row(h, W_DKV, W_KR, pos, base, kv_norm_weight=None, kv_norm_eps=1e-5):
    r = O.cache_rows(h, W_DKV, W_KR, pos, base)
    if kv_norm_weight is None:
        return r
    w = np.concatenate([kv_norm_weight, np.ones(r.shape[1] - len(kv_norm_weight))])
    return O.rms_norm(r, w, kv_norm_eps)


@pytest.mark.parametrize("mutant", [_rms_norm_sum_not_mean, _rms_norm_eps_outside])
def test_planted_rms_norm_mistakes_are_caught(mutant):
    assert not check_rms_norm(mutant)


def test_planted_kv_norm_row_mistake_is_caught():
    assert not check_cache_rows_kv_norm(_cache_rows_norm_whole_row)


# ---------------------------------------------------------------------------
# pins: the pre-merged weight forms (MLA page §4)
# ---------------------------------------------------------------------------
def check_premerged_query(fn):
    """Brute-force triple loop on tiny shapes; the merged map reaches the
    two-step absorbed query; each head's merged map has rank <= d_h."""
    rng = np.random.default_rng(31)
    n_h, d_h, d_c, d_cq = 3, 2, 5, 4
    W_UQ = rng.standard_normal((n_h * d_h, d_cq))
    W_UK = rng.standard_normal((n_h * d_h, d_c))
    got = np.asarray(fn(W_UQ, W_UK, n_h, d_h))
    if got.shape != (n_h, d_c, d_cq):
        return False
    ok = True
    for i in range(n_h):
        for c in range(d_c):
            for q in range(d_cq):
                ref = sum(W_UK[i * d_h + k, c] * W_UQ[i * d_h + k, q] for k in range(d_h))
                ok &= abs(got[i, c, q] - ref) <= 1e-12
    # W_QK_i c_Q equals the absorbed query's latent part q~_i = W_UK_i^T (W_UQ_i c_Q)
    m = MICRO
    W, _, h_new = micro_inputs(32, L=3)
    q_abs, parts = O.absorbed_query(h_new, W["W_DQ"], W["W_UQ"], W["W_QR"], W["W_UK"], np.array([3]),
                                    m["n_h"], m["d_h"], m["d_r"], 10000.0, return_parts=True)
    WQK = fn(W["W_UQ"], W["W_UK"], m["n_h"], m["d_h"])
    ok &= np.allclose(np.einsum("icq,bq->bic", WQK, parts["c_Q"]), q_abs[..., :m["d_c"]], rtol=1e-12, atol=1e-12)
    W_UQ = rng.standard_normal((2 * 3, 9))
    W_UK = rng.standard_normal((2 * 3, 8))
    for Wi in fn(W_UQ, W_UK, 2, 3):
        sv = np.linalg.svd(Wi, compute_uv=False)
        ok &= bool(np.all(sv[3:] <= 1e-10 * sv[0]))
    return bool(ok)


def check_premerged_output(fn):
    """Brute-force loop on tiny shapes; the merged map reaches the two-step
    output projection."""
    rng = np.random.default_rng(33)
    n_h, d_h, d_c, d = 3, 2, 4, 5
    W_UV = rng.standard_normal((n_h * d_h, d_c))
    W_O = rng.standard_normal((d, n_h * d_h))
    got = np.asarray(fn(W_UV, W_O, n_h, d_h))
    if got.shape != (d, n_h * d_c):
        return False
    ok = True
    for r in range(d):
        for i in range(n_h):
            for c in range(d_c):
                ref = sum(W_O[r, i * d_h + k] * W_UV[i * d_h + k, c] for k in range(d_h))
                ok &= abs(got[r, i * d_c + c] - ref) <= 1e-12
    o_lat = rng.standard_normal((2, n_h, d_c))
    ok &= np.allclose(o_lat.reshape(2, -1) @ got.T, O.output_projection(o_lat, W_UV, W_O, n_h, d_h),
                      rtol=1e-12, atol=1e-12)
    return bool(ok)


def test_premerged_query_weights():
    assert check_premerged_query(O.premerged_query_weights)


def test_premerged_output_weights():
    assert check_premerged_output(O.premerged_output_weights)


def _premerged_query_transposed(W_UQ, W_UK, n_h, d_h):
    # W_UQ_i^T W_UK_i, the score's bilinear form, instead of the map applied to c_Q
    return np.transpose(O.premerged_query_weights(W_UQ, W_UK, n_h, d_h), (0, 2, 1))


def _premerged_query_head_mixed(W_UQ, W_UK, n_h, d_h):
    W = O.premerged_query_weights(W_UQ, W_UK, n_h, d_h)
    return np.roll(W, 1, axis=0)


def _premerged_output_blocks_swapped(W_UV, W_O, n_h, d_h):
    W = O.premerged_output_weights(W_UV, W_O, n_h, d_h)
    d_c = np.asarray(W_UV).shape[1]
    return np.concatenate([W[:, d_c:2 * d_c], W[:, :d_c], W[:, 2 * d_c:]], axis=1)


@pytest.mark.parametrize("mutant", [_premerged_query_transposed, _premerged_query_head_mixed])
def test_planted_premerged_query_mistakes_are_caught(mutant):
    assert not check_premerged_query(mutant)


def test_planted_premerged_output_mistake_is_caught():
    assert not check_premerged_output(_premerged_output_blocks_swapped)


# ---------------------------------------------------------------------------
# pins: the materialised (MHA) path for several new tokens (Latent page: prefill
# takes the MHA path; MiniMind page §10 naive version, §12 causal visibility)
# ---------------------------------------------------------------------------
def check_mha_brute(fn):
    """Pure-Python loops on tiny shapes, including rows that a query must not see."""
    rng = np.random.default_rng(41)
    T, L, n_h, d_h, d_r = 3, 6, 2, 3, 2
    q = rng.standard_normal((T, n_h, d_h + d_r))
    k_c = rng.standard_normal((L, n_h, d_h))
    k_r = rng.standard_normal((L, d_r))
    v_c = rng.standard_normal((L, n_h, d_h))
    q_pos = np.array([2, 3, 5])
    sc = 0.6
    o, lse = fn(q, k_c, k_r, v_c, q_pos, sc)
    ok = True
    for t in range(T):
        for i in range(n_h):
            s = [sc * (sum(q[t, i, c] * k_c[r, i, c] for c in range(d_h)) +
                       sum(q[t, i, d_h + c] * k_r[r, c] for c in range(d_r))) for r in range(q_pos[t] + 1)]
            ref_lse = logsumexp(s)
            w = [math.exp(v - ref_lse) for v in s]
            ref_o = [sum(w[r] * v_c[r, i, c] for r in range(len(s))) for c in range(d_h)]
            ok &= abs(lse[t, i] - ref_lse) < 1e-12 and np.allclose(o[t, i], ref_o, rtol=1e-12, atol=1e-14)
    return bool(ok)


def check_prefill_rows_are_decode_steps(prefill):
    """Row t of a T-token prefill equals the decode step of new token t with the
    context and new tokens 0..t-1 cached (the decode definition is pinned above)."""
    m = MICRO
    W, h_ctx, _ = micro_inputs(42, L=4)
    rng = np.random.default_rng(43)
    h_new = rng.standard_normal((3, m["d"]))
    us, os_, lses = prefill([h_ctx[0]], [h_new], W, m["n_h"], m["d_h"], m["d_r"], 10000.0, return_parts=True)
    ok = True
    for t in range(3):
        ctx = np.concatenate([h_ctx[0], h_new[:t]])
        u, o, lse = O.decode_materialised([ctx], h_new[t:t + 1], W, m["n_h"], m["d_h"], m["d_r"], 10000.0,
                                          return_parts=True)
        ok &= np.allclose(us[0][t], u[0], rtol=1e-10, atol=1e-12) and np.allclose(os_[0][t], o[0], rtol=1e-10,
                                                                                   atol=1e-12)
        ok &= np.allclose(lses[0][t], lse[0], rtol=1e-12, atol=1e-12)
    return bool(ok)


def check_prefill_causal(prefill):
    """Changing the last new token leaves every earlier row unchanged."""
    m = MICRO
    W, h_ctx, _ = micro_inputs(44, L=2)
    rng = np.random.default_rng(45)
    h_new = rng.standard_normal((4, m["d"]))
    h_alt = h_new.copy()
    h_alt[-1] += 3.0
    a = prefill([h_ctx[0]], [h_new], W, m["n_h"], m["d_h"], m["d_r"], 10000.0)[0]
    b = prefill([h_ctx[0]], [h_alt], W, m["n_h"], m["d_h"], m["d_r"], 10000.0)[0]
    return bool(np.allclose(a[:-1], b[:-1], rtol=1e-13, atol=1e-13) and not np.allclose(a[-1], b[-1]))


def test_mha_attention_brute_force():
    assert check_mha_brute(O.mha_attention)


def test_prefill_rows_are_decode_steps():
    assert check_prefill_rows_are_decode_steps(O.prefill_materialised)


def test_prefill_is_causal():
    assert check_prefill_causal(O.prefill_materialised)


def test_materialised_query_is_absorbed_query_parts():
    m = MICRO
    W, _, h_new = micro_inputs(46, L=2)
    pos = np.array([7])
    q = O.materialised_query(h_new, W["W_DQ"], W["W_UQ"], W["W_QR"], pos, m["n_h"], m["d_h"], m["d_r"], 10000.0)
    _, parts = O.absorbed_query(h_new, W["W_DQ"], W["W_UQ"], W["W_QR"], W["W_UK"], pos, m["n_h"], m["d_h"], m["d_r"],
                                10000.0, return_parts=True)
    assert np.allclose(q, np.concatenate([parts["q_C"], parts["q_R"]], axis=-1), rtol=1e-13, atol=1e-13)


_MHA = O.mha_attention


def _mha_no_mask(q, k_c, k_r, v_c, q_pos, scale):
    return _MHA(q, k_c, k_r, v_c, np.full(len(q_pos), np.asarray(k_c).shape[0] - 1), scale)


def _mha_excludes_self(q, k_c, k_r, v_c, q_pos, scale):
    return _MHA(q, k_c, k_r, v_c, np.asarray(q_pos) - 1, scale)


def _prefill_with(mha):
    def run(h_ctx_list, h_new_list, W, n_h, d_h, d_r, base, return_parts=False):
        orig = O.mha_attention
        O.mha_attention = mha
        try:
            return O.prefill_materialised(h_ctx_list, h_new_list, W, n_h, d_h, d_r, base, return_parts)
        finally:
            O.mha_attention = orig
    return run


@pytest.mark.parametrize("mutant", [_mha_no_mask, _mha_excludes_self])
def test_planted_mha_mistakes_are_caught(mutant):
    assert not check_mha_brute(mutant)
    assert not (check_prefill_rows_are_decode_steps(_prefill_with(mutant))
                and check_prefill_causal(_prefill_with(mutant)))
