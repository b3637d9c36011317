"""Parity of every entry point of the CUDA library against the fp64 oracle,
element by element, on seeded generator inputs (never on another stage's GPU
output). Sizes span several tiles and ragged tails; the full-size workloads are
checked on sampled sequences the oracle can compute."""
import numpy as np
import pytest

import mla_synth as S
from oracle import mla as O
from gpu_helpers import (TOL, TOL_E2E, TOL_LSE_E2E, TOL_LSE_E2E_MANY, assert_close, dev, dev_i32, host, make_weights_dev, decoder,
                         torch_dtype)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)
import head_latent_attention_24_b300 as M  # noqa: E402

SMALL = ["tiny", "minimind", "v2"]
# Projection kernel families: the tensor-core kernel (AUTO for bf16) and the
# CUDA-core kernel (forced). fp32 layers always take the CUDA-core kernel.
PROJ = ["auto", "simt"]


def set_proj(dec, proj):
    M.mla_set_proj_path(dec.handle, M.MLA_PROJ_SIMT if proj == "simt" else M.MLA_PROJ_AUTO)


def small_shape(name, batch=None, ctx=None):
    shp = S.workload(name)
    if name == "tiny":
        return shp
    return shp.scaled(batch=batch or 3, ctx=ctx or 301)


# --------------------------------------------------------------------- S1
@pytest.mark.parametrize("name", SMALL)
@pytest.mark.parametrize("proj", PROJ)
@pytest.mark.parametrize("n", [150, 600])
def test_append_matches_oracle_and_touches_only_its_rows(name, proj, n):
    # n = 600 spans three 256-row tiles of the tensor-core kernel with a ragged tail
    shp = small_shape(name)
    W = S.draw_weights(shp)
    B, L = 3, 250
    rng = np.random.default_rng(1)
    # distinct rows, the first one at the last position of the last sequence
    flat = np.concatenate([[B * L - 1], rng.choice(B * L - 1, size=n - 1, replace=False)])
    seq, pos = flat // L, flat % L
    x = S.draw_context_h(shp, 0, n)
    dec = decoder(shp, make_weights_dev(shp, W), B, L)
    set_proj(dec, proj)
    cache = torch.full((B, L, shp.D), float("nan"), dtype=torch_dtype(shp), device="cuda")
    dec.append(dev(x, shp), dev_i32(seq), dev_i32(pos), cache)
    st, bits = M.mla_get_device_status(dec.handle)
    assert st == M.MLA_OK and bits == 0
    got = host(cache)
    ref = O.cache_rows(x, W["W_DKV"], W["W_KR"], pos, shp.rope_base)
    assert_close(got[seq, pos], ref, shp.dtype, what="cache rows")
    untouched = np.ones((B, L), bool)
    untouched[seq, pos] = False
    assert np.isnan(got[untouched]).all()


@pytest.mark.parametrize("name", SMALL)
@pytest.mark.parametrize("proj", PROJ)
def test_append_bit_exact_on_integer_inputs(name, proj):
    # Integer h and weights: every product and fp32 sum is exact, so after one
    # rounding to the storage dtype the cache must equal the oracle bit for bit.
    # Position 0 makes RoPE the identity; c_KV is exact at any position.
    shp = small_shape(name)
    rng = np.random.default_rng(2)
    W = {k: rng.integers(-3, 4, size=shp.weight_shape(k)).astype(np.float64) for k in S.WEIGHT_NAMES}
    n, B, L = 40, 4, 16
    x = rng.integers(-3, 4, size=(n, shp.d)).astype(np.float64)
    seq = np.arange(n) % B
    pos = np.where(np.arange(n) < B, 0, 1 + np.arange(n) // B)
    dec = decoder(shp, make_weights_dev(shp, W), B, L)
    set_proj(dec, proj)
    cache = torch.zeros((B, L, shp.D), dtype=torch_dtype(shp), device="cuda")
    dec.append(dev(x, shp), dev_i32(seq), dev_i32(pos), cache)
    got = host(cache)[seq, pos]
    ref = S.to_dtype(O.cache_rows(x, W["W_DKV"], W["W_KR"], pos, shp.rope_base), shp.dtype)
    assert np.array_equal(got[:, :shp.d_c], ref[:, :shp.d_c])
    at0 = pos == 0
    assert np.array_equal(got[at0], ref[at0])


def test_append_out_of_range_rows_are_skipped_and_flagged():
    shp = S.workload("tiny")
    W = S.draw_weights(shp)
    B, L = 2, 8
    x = S.draw_context_h(shp, 0, 4)
    dec = decoder(shp, make_weights_dev(shp, W), B, L)
    cache = torch.zeros((B, L, shp.D), dtype=torch_dtype(shp), device="cuda")
    dec.append(dev(x, shp), dev_i32([0, 5, 1, 0]), dev_i32([0, 1, 9, -1]), cache)
    st, bits = M.mla_get_device_status(dec.handle)
    assert st == M.MLA_ERR_DEVICE
    assert bits & M.MLA_DEV_SEQ_RANGE and bits & M.MLA_DEV_POS_RANGE
    got = host(cache)
    ref = O.cache_rows(x[:1], W["W_DKV"], W["W_KR"], [0], shp.rope_base)
    assert_close(got[0, 0:1], ref, shp.dtype)
    got[0, 0] = 0
    assert np.all(got == 0)
    assert M.mla_get_device_status(dec.handle) == (M.MLA_OK, 0)   # cleared by the read


# --------------------------------------------------------------------- S2
@pytest.mark.parametrize("name", SMALL)
@pytest.mark.parametrize("proj", PROJ)
def test_absorb_q_matches_oracle(name, proj):
    shp = small_shape(name)
    W = S.draw_weights(shp)
    B = 37 if name != "tiny" else 2
    h = S.draw_new_tokens(shp, B)
    max_pos = 5000
    pos = np.random.default_rng(3).integers(0, max_pos, size=B)
    pos[0], pos[-1] = 0, max_pos - 1
    dec = decoder(shp, make_weights_dev(shp, W), B, 16, max_pos=max_pos)
    set_proj(dec, proj)
    M.mla_absorb_q(dec.handle, dev(h, shp), B, dec.W["W_DQ"], dec.W["W_UQ"], dec.W["W_QR"], dec.W["W_UK"],
                   dev_i32(pos), dec.q_abs, dec.ws, dec.ws.numel())
    ref = O.absorbed_query(h, W["W_DQ"], W["W_UQ"], W["W_QR"], W["W_UK"], pos, shp.n_h, shp.d_h, shp.d_r,
                           shp.rope_base)
    got = host(dec.q_abs)
    assert_close(got, ref, shp.dtype, what="q_abs")
    assert M.mla_get_device_status(dec.handle) == (M.MLA_OK, 0)


# --------------------------------------------------------------------- S3
def run_decode(shp, q_abs, rows_per_seq, seqlens, max_len, path=None):
    B = len(seqlens)
    cache = np.zeros((B, max_len, shp.D))
    for b, r in enumerate(rows_per_seq):
        cache[b, :len(r)] = r
    W = {k: np.zeros(shp.weight_shape(k)) for k in S.WEIGHT_NAMES}
    dec = decoder(shp, {k: torch.zeros(1, device="cuda") for k in W}, B, max_len)
    if path is not None:
        M.mla_set_decode_path(dec.handle, path)
    M.mla_decode_attn(dec.handle, dev(q_abs, shp), dev(cache, shp), B, max_len, dev_i32(seqlens), dec.o_lat,
                      dec.lse, dec.ws, dec.ws.numel())
    st, bits = M.mla_get_device_status(dec.handle)
    return host(dec.o_lat), dec.lse.cpu().numpy().astype(np.float64), st, bits, dec


def oracle_decode(shp, q_abs, rows_per_seq, seqlens):
    sc = O.scale_of(shp.d_h, shp.d_r)
    outs = [O.latent_attention(q_abs[b], rows_per_seq[b][:seqlens[b]], shp.d_c, sc) for b in range(len(seqlens))]
    return np.stack([o for o, _ in outs]), np.stack([l for _, l in outs])


SEQLEN_PATTERNS = {
    "uniform": lambda rng, L: np.full(5, L),
    "ragged": lambda rng, L: np.array([1, L, 0, 33, L // 2 + 7, 64, 65, 2]),
}


def paths():
    return [None, M.MLA_DECODE_SIMT]


@pytest.mark.parametrize("name", ["minimind", "v2"])
@pytest.mark.parametrize("chunks", [1, 3, 40, 200])
def test_decode_attn_any_chunk_count(name, chunks):
    """Split-KV with a forced chunk count, from one chunk for the whole batch
    to 64-row slivers (a 700-row sequence then spans 11 chunks and the merge
    takes 11 partials; most of the 200 chunks are empty): matches the oracle."""
    shp = S.workload(name)
    max_len = 700
    seqlens = np.array([700, 1, 0, 333, 690])
    B = len(seqlens)
    q = S.draw_absorbed_queries(shp, B)
    rows = [S.draw_latent_rows(shp, int(seqlens[b]), sub=b) for b in range(B)]
    ref_o, ref_l = oracle_decode(shp, q, rows, seqlens)
    cache = np.zeros((B, max_len, shp.D))
    for b, r in enumerate(rows):
        cache[b, :len(r)] = r
    dec = decoder(shp, {k: torch.zeros(1, device="cuda") for k in S.WEIGHT_NAMES}, B, max_len)
    M.mla_set_decode_chunks(dec.handle, chunks)
    ws = torch.empty(M.mla_decode_workspace_size(dec.handle, B, max_len), dtype=torch.uint8, device="cuda")
    M.mla_decode_attn(dec.handle, dev(q, shp), dev(cache, shp), B, max_len, dev_i32(seqlens), dec.o_lat, dec.lse,
                      ws, ws.numel())
    st, bits = M.mla_get_device_status(dec.handle)
    assert st == M.MLA_OK and bits == 0
    got_o, got_l = host(dec.o_lat), dec.lse.cpu().numpy().astype(np.float64)
    nz = seqlens > 0
    assert_close(got_o[nz], ref_o[nz], shp.dtype, what="o_lat")
    assert np.all(got_o[~nz] == 0) and np.all(np.isneginf(got_l[~nz]))
    assert np.abs(got_l[nz] - ref_l[nz]).max() <= 2e-4 * max(1, np.abs(ref_l[nz]).max())
    dec.close()


@pytest.mark.parametrize("B", [507, 508, 900])
def test_decode_attn_many_short_sequences(B):
    """Batches around and past the size whose split plan the few-head kernel
    works out in its own shared memory (up to 507 sequences; larger batches
    take the separate plan launch): short ragged sequences, some empty, against
    the oracle."""
    shp = S.workload("minimind")
    max_len = 40
    seqlens = np.random.default_rng(B).integers(0, max_len + 1, size=B)
    seqlens[:3] = [0, 1, max_len]
    q = S.draw_absorbed_queries(shp, B)
    rows = [S.draw_latent_rows(shp, int(seqlens[b]), sub=b) for b in range(B)]
    ref_o, ref_l = oracle_decode(shp, q, rows, seqlens)
    got_o, got_l, st, bits, dec = run_decode(shp, q, rows, seqlens, max_len)
    assert M.mla_get_decode_path(dec.handle) == M.MLA_DECODE_TCGEN05
    assert M.mla_last_launch_count(dec.handle) == (2 if B <= 507 else 3)
    assert st == M.MLA_OK and bits == 0
    nz = seqlens > 0
    assert_close(got_o[nz], ref_o[nz], shp.dtype, what="o_lat")
    assert np.all(got_o[~nz] == 0) and np.all(np.isneginf(got_l[~nz]))
    assert np.abs(got_l[nz] - ref_l[nz]).max() <= 2e-4 * max(1, np.abs(ref_l[nz]).max())
    dec.close()


@pytest.mark.parametrize("name", SMALL)
@pytest.mark.parametrize("pattern", list(SEQLEN_PATTERNS))
def test_decode_attn_matches_oracle(name, pattern):
    shp = S.workload(name)
    max_len = 301 if name != "tiny" else 129
    seqlens = SEQLEN_PATTERNS[pattern](np.random.default_rng(4), max_len)
    B = len(seqlens)
    q = S.draw_absorbed_queries(shp, B)
    rows = [S.draw_latent_rows(shp, int(seqlens[b]), sub=b) for b in range(B)]
    ref_o, ref_l = oracle_decode(shp, q, rows, seqlens)
    got_o, got_l, st, bits, _ = run_decode(shp, q, rows, seqlens, max_len)
    assert st == M.MLA_OK and bits == 0
    nz = seqlens > 0
    assert_close(got_o[nz], ref_o[nz], shp.dtype, what="o_lat")
    assert np.all(got_o[~nz] == 0) and np.all(np.isneginf(got_l[~nz]))
    assert np.abs(got_l[nz] - ref_l[nz]).max() <= (2e-5 if shp.dtype == "f32" else 2e-4) * max(1, np.abs(ref_l[nz]).max())


@pytest.mark.parametrize("name", SMALL)
def test_decode_attn_special_cases(name):
    shp = S.workload(name)
    max_len = 97
    B = 3
    q = S.draw_absorbed_queries(shp, B)
    one = S.draw_latent_rows(shp, 1, sub=7)
    same = np.tile(S.draw_latent_rows(shp, 1, sub=8), (max_len, 1))
    rows = [one, same, S.draw_latent_rows(shp, max_len, sub=9)]
    q[2] = 0.0
    seqlens = np.array([1, max_len, max_len])
    got_o, got_l, st, bits, _ = run_decode(shp, q, rows, seqlens, max_len)
    sc = O.scale_of(shp.d_h, shp.d_r)
    # seqlen 1: the only row's latent, exactly; lse = its score
    assert np.array_equal(got_o[0], np.broadcast_to(one[0, :shp.d_c], (shp.n_h, shp.d_c)))
    assert np.allclose(got_l[0], sc * q[0] @ one[0], rtol=1e-5, atol=1e-5)
    # all rows equal: that row. Exact for bf16 storage (the fp32 result rounds
    # back onto the row's bf16 values); for fp32 storage a sequence split
    # across chunks is merged by weights that sum to one only up to fp32 rounding.
    want = np.broadcast_to(same[0, :shp.d_c], (shp.n_h, shp.d_c))
    if shp.dtype == "bf16":
        assert np.array_equal(got_o[1], want)
    else:
        assert np.allclose(got_o[1], want, rtol=2e-6, atol=0)
    # q = 0: the mean of the rows, lse = log(L)
    assert_close(got_o[2], np.broadcast_to(rows[2][:, :shp.d_c].mean(0), (shp.n_h, shp.d_c)), shp.dtype)
    assert np.allclose(got_l[2], np.log(max_len), rtol=1e-6)


@pytest.mark.parametrize("name", SMALL)
@pytest.mark.parametrize("direction", ["rising", "falling"])
def test_decode_attn_monotone_scores(name, direction):
    # Scores that climb by ~12 (base 2) per 64 rows move the running maximum on
    # every tile, so the online softmax must rescale its accumulator each time;
    # falling scores keep the first tile's maximum throughout.
    shp = S.workload(name)
    max_len = 700
    seqlens = np.array([700, 333, 64, 65])
    B = len(seqlens)
    sc = O.scale_of(shp.d_h, shp.d_r)
    q = np.zeros((B, shp.n_h, shp.D))
    q[:, :, 0] = S.to_dtype(np.linspace(0.5, 1.0, shp.n_h), shp.dtype)
    rows = []
    for b, n in enumerate(seqlens):
        r = S.draw_latent_rows(shp, int(n), sub=40 + b) * 0.25
        t = np.arange(n) if direction == "rising" else (n - 1 - np.arange(n))
        r[:, 0] = S.to_dtype(t * (12.0 / 64.0) / np.log2(np.e) / sc, shp.dtype)
        rows.append(S.to_dtype(r, shp.dtype))
    ref_o, ref_l = oracle_decode(shp, q, rows, seqlens)
    got_o, got_l, st, bits, _ = run_decode(shp, q, rows, seqlens, max_len)
    assert st == M.MLA_OK and bits == 0
    assert_close(got_o, ref_o, shp.dtype, what="o_lat")
    assert np.abs(got_l - ref_l).max() <= (2e-5 if shp.dtype == "f32" else 2e-4) * max(1, np.abs(ref_l).max())


# Sequence layouts that give every chunk of the split-KV plan several
# 128-row tiles (the other cases mostly give one tile per chunk): whole
# sequences of 3 tiles per chunk, one long sequence split over every chunk,
# and lengths that end mid-tile.
LONG_LAYOUTS = {
    "3_tiles_whole": lambda: np.full(74, 384),
    "1_seq_split": lambda: np.array([74 * 384]),
    "ragged_tails": lambda: np.array([5000, 4097, 333, 64 * 75 + 1]),
}


@pytest.mark.parametrize("layout", list(LONG_LAYOUTS))
def test_decode_attn_multi_tile_chunks(layout):
    shp = S.workload("v2")
    seqlens = LONG_LAYOUTS[layout]()
    B, max_len = len(seqlens), int(seqlens.max())
    q = S.draw_absorbed_queries(shp, B)
    rows = [S.draw_latent_rows(shp, int(n), sub=60 + b) for b, n in enumerate(seqlens)]
    ref_o, ref_l = oracle_decode(shp, q, rows, seqlens)
    got_o, got_l, st, bits, _ = run_decode(shp, q, rows, seqlens, max_len)
    assert st == M.MLA_OK and bits == 0
    assert np.abs(got_l - ref_l).max() <= 2e-4 * max(1, np.abs(ref_l).max())
    assert_close(got_o, ref_o, shp.dtype, what="o_lat")


def test_decode_attn_equal_rows_long():
    # Every row of a sequence equal: o_lat is that row whatever the weights,
    # as long as the weights applied to the rows are the ones summed into the
    # softmax denominator. Several tiles per chunk.
    shp = S.workload("v2")
    seqlens = np.array([9000, 7000])
    B, max_len = 2, 9000
    q = S.draw_absorbed_queries(shp, B)
    rows = [np.tile(S.draw_latent_rows(shp, 1, sub=70 + b), (int(n), 1)) for b, n in enumerate(seqlens)]
    got_o, got_l, st, bits, _ = run_decode(shp, q, rows, seqlens, max_len)
    assert st == M.MLA_OK and bits == 0
    for b in range(B):
        want = np.broadcast_to(rows[b][0, :shp.d_c], (shp.n_h, shp.d_c))
        assert_close(got_o[b], want, shp.dtype, what=f"o_lat[{b}]")


def test_decode_attn_clamps_and_flags_bad_seqlens():
    shp = S.workload("minimind")
    max_len = 50
    q = S.draw_absorbed_queries(shp, 2)
    rows = [S.draw_latent_rows(shp, max_len, sub=b) for b in range(2)]
    got_o, got_l, st, bits, _ = run_decode(shp, q, rows, np.array([max_len + 9, -3]), max_len)
    assert st == M.MLA_ERR_DEVICE and bits & M.MLA_DEV_SEQLEN_RANGE
    ref_o, ref_l = oracle_decode(shp, q, rows, np.array([max_len, 0]))
    assert_close(got_o[0], ref_o[0], shp.dtype)
    assert np.all(got_o[1] == 0) and np.isneginf(got_l[1]).all()


def test_decode_attn_paths_agree():
    shp = S.workload("v2")
    max_len = 700
    seqlens = np.array([700, 129, 1, 640])
    q = S.draw_absorbed_queries(shp, 4)
    rows = [S.draw_latent_rows(shp, int(n), sub=b) for b, n in enumerate(seqlens)]
    a = run_decode(shp, q, rows, seqlens, max_len, path=M.MLA_DECODE_SIMT)
    b = run_decode(shp, q, rows, seqlens, max_len, path=M.MLA_DECODE_AUTO)
    assert_close(b[0], a[0], "bf16")


def test_workspace_and_alignment_errors():
    shp = S.workload("tiny")
    q = S.draw_absorbed_queries(shp, 2)
    rows = [S.draw_latent_rows(shp, 10, sub=b) for b in range(2)]
    _, _, _, _, dec = run_decode(shp, q, rows, np.array([10, 10]), 10)
    qd, cd = dev(q, shp), torch.zeros((2, 10, shp.D), dtype=torch.float32, device="cuda")
    sl = dev_i32([10, 10])
    with pytest.raises(M.MLAError) as e:
        M.mla_decode_attn(dec.handle, qd, cd, 2, 10, sl, dec.o_lat, dec.lse, dec.ws, 16)
    assert e.value.status == M.MLA_ERR_WORKSPACE
    with pytest.raises(M.MLAError) as e:
        M.mla_decode_attn(dec.handle, qd.data_ptr() + 4, cd, 2, 10, sl, dec.o_lat, dec.lse, dec.ws, dec.ws.numel())
    assert e.value.status == M.MLA_ERR_INVALID_ARG


# --------------------------------------------------------------------- S4/S5
@pytest.mark.parametrize("name", SMALL)
@pytest.mark.parametrize("proj", PROJ)
def test_out_proj_matches_oracle(name, proj):
    shp = small_shape(name)
    W = S.draw_weights(shp)
    B = 19 if name != "tiny" else 2
    o_lat = S.to_dtype(S.draw_latent_rows(shp, B * shp.n_h, sub=11)[:, :shp.d_c].reshape(B, shp.n_h, shp.d_c)
                       / 8.0, shp.dtype)
    dec = decoder(shp, make_weights_dev(shp, W), B, 16)
    set_proj(dec, proj)
    M.mla_out_proj(dec.handle, dev(o_lat, shp), B, dec.W["W_UV"], dec.W["W_O"], dec.u, dec.ws, dec.ws.numel())
    ref = O.output_projection(o_lat, W["W_UV"], W["W_O"], shp.n_h, shp.d_h)
    assert_close(host(dec.u), ref, shp.dtype, what="u")


@pytest.mark.parametrize("name", ["minimind", "v2"])
def test_projections_full_size(name):
    """The benchmark's projection shapes (batch 256 for MiniMind, 64 for V2, the
    full layer widths), in the launch configuration the benchmark uses: new-token
    cache rows, the absorbed query and the output projection against the oracle."""
    shp = S.workload(name)
    W = S.draw_weights(shp)
    B = shp.batch
    h = S.draw_new_tokens(shp, B)
    pos = np.random.default_rng(5).integers(0, 4097, size=B)
    dec = decoder(shp, make_weights_dev(shp, W), B, 4097, max_pos=4097)
    cache = torch.full((B, 4097, shp.D), float("nan"), dtype=torch_dtype(shp), device="cuda")
    M.mla_append_cache(dec.handle, dev(h, shp), B, dec.W["W_DKV"], dec.W["W_KR"], dec.tok_seq, dev_i32(pos), cache,
                       B, 4097)
    M.mla_absorb_q(dec.handle, dev(h, shp), B, dec.W["W_DQ"], dec.W["W_UQ"], dec.W["W_QR"], dec.W["W_UK"],
                   dev_i32(pos), dec.q_abs, dec.ws, dec.ws.numel())
    o_lat = S.to_dtype(S.draw_latent_rows(shp, B * shp.n_h, sub=12)[:, :shp.d_c].reshape(B, shp.n_h, shp.d_c)
                       / 8.0, shp.dtype)
    M.mla_out_proj(dec.handle, dev(o_lat, shp), B, dec.W["W_UV"], dec.W["W_O"], dec.u, dec.ws, dec.ws.numel())
    assert M.mla_get_device_status(dec.handle) == (M.MLA_OK, 0)
    got_rows = host(cache)[np.arange(B), pos]
    assert_close(got_rows, O.cache_rows(h, W["W_DKV"], W["W_KR"], pos, shp.rope_base), shp.dtype, what="cache rows")
    ref_q = O.absorbed_query(h, W["W_DQ"], W["W_UQ"], W["W_QR"], W["W_UK"], pos, shp.n_h, shp.d_h, shp.d_r,
                             shp.rope_base)
    assert_close(host(dec.q_abs), ref_q, shp.dtype, what="q_abs")
    ref_u = O.output_projection(o_lat, W["W_UV"], W["W_O"], shp.n_h, shp.d_h)
    assert_close(host(dec.u), ref_u, shp.dtype, what="u")


# --------------------------------------------------------------------- pre-merged forms
def premerged_dev(shp, dec):
    """The library's merged weights for the decoder's weights (setup calls)."""
    dt = torch_dtype(shp)
    W_QK = torch.empty((shp.n_h, shp.d_c, shp.d_cq), dtype=dt, device="cuda")
    W_OUV = torch.empty((shp.d, shp.n_h * shp.d_c), dtype=dt, device="cuda")
    M.mla_premerge_query_weights(dec.handle, dec.W["W_UQ"], dec.W["W_UK"], W_QK)
    M.mla_premerge_output_weights(dec.handle, dec.W["W_UV"], dec.W["W_O"], W_OUV)
    return W_QK, W_OUV


@pytest.mark.parametrize("name", SMALL)
def test_premerged_weights_match_oracle(name):
    shp = small_shape(name)
    W = S.draw_weights(shp)
    dec = decoder(shp, make_weights_dev(shp, W), 2, 16)
    W_QK, W_OUV = premerged_dev(shp, dec)
    ref_qk = O.premerged_query_weights(W["W_UQ"], W["W_UK"], shp.n_h, shp.d_h)
    ref_ouv = O.premerged_output_weights(W["W_UV"], W["W_O"], shp.n_h, shp.d_h)
    assert_close(host(W_QK), ref_qk, shp.dtype, what="W_QK")
    assert_close(host(W_OUV), ref_ouv, shp.dtype, what="W_OUV")


@pytest.mark.parametrize("name", SMALL)
@pytest.mark.parametrize("proj", PROJ)
def test_premerged_calls_match_oracle(name, proj):
    """The absorbed query through W_QK and the output through W_OUV reach the
    oracle's two-step forms (the merge is exact up to rounding)."""
    shp = small_shape(name)
    W = S.draw_weights(shp)
    B = 37 if name != "tiny" else 2
    h = S.draw_new_tokens(shp, B)
    max_pos = 5000
    pos = np.random.default_rng(7).integers(0, max_pos, size=B)
    pos[0], pos[-1] = 0, max_pos - 1
    dec = decoder(shp, make_weights_dev(shp, W), B, 16, max_pos=max_pos)
    set_proj(dec, proj)
    W_QK, W_OUV = premerged_dev(shp, dec)
    M.mla_absorb_q_premerged(dec.handle, dev(h, shp), B, dec.W["W_DQ"], W_QK, dec.W["W_QR"], dev_i32(pos),
                             dec.q_abs, dec.ws, dec.ws.numel())
    ref_q = O.absorbed_query(h, W["W_DQ"], W["W_UQ"], W["W_QR"], W["W_UK"], pos, shp.n_h, shp.d_h, shp.d_r,
                             shp.rope_base)
    assert_close(host(dec.q_abs), ref_q, shp.dtype, what="q_abs (pre-merged)")
    o_lat = S.to_dtype(S.draw_latent_rows(shp, B * shp.n_h, sub=13)[:, :shp.d_c].reshape(B, shp.n_h, shp.d_c)
                       / 8.0, shp.dtype)
    M.mla_out_proj_premerged(dec.handle, dev(o_lat, shp), B, W_OUV, dec.u)
    ref_u = O.output_projection(o_lat, W["W_UV"], W["W_O"], shp.n_h, shp.d_h)
    assert_close(host(dec.u), ref_u, shp.dtype, what="u (pre-merged)")
    assert M.mla_get_device_status(dec.handle) == (M.MLA_OK, 0)


def test_premerged_full_size_v2():
    """The benchmark's V2 projection shapes (batch 64) through the pre-merged maps."""
    shp = S.workload("v2")
    W = S.draw_weights(shp)
    B = shp.batch
    h = S.draw_new_tokens(shp, B)
    pos = np.random.default_rng(9).integers(0, 4097, size=B)
    dec = decoder(shp, make_weights_dev(shp, W), B, 4097, max_pos=4097)
    W_QK, W_OUV = premerged_dev(shp, dec)
    M.mla_absorb_q_premerged(dec.handle, dev(h, shp), B, dec.W["W_DQ"], W_QK, dec.W["W_QR"], dev_i32(pos),
                             dec.q_abs, dec.ws, dec.ws.numel())
    assert M.mla_last_launch_count(dec.handle) == 2
    o_lat = S.to_dtype(S.draw_latent_rows(shp, B * shp.n_h, sub=14)[:, :shp.d_c].reshape(B, shp.n_h, shp.d_c)
                       / 8.0, shp.dtype)
    M.mla_out_proj_premerged(dec.handle, dev(o_lat, shp), B, W_OUV, dec.u)
    assert M.mla_last_launch_count(dec.handle) == 1
    assert M.mla_get_device_status(dec.handle) == (M.MLA_OK, 0)
    ref_q = O.absorbed_query(h, W["W_DQ"], W["W_UQ"], W["W_QR"], W["W_UK"], pos, shp.n_h, shp.d_h, shp.d_r,
                             shp.rope_base)
    assert_close(host(dec.q_abs), ref_q, shp.dtype, what="q_abs (pre-merged)")
    ref_u = O.output_projection(o_lat, W["W_UV"], W["W_O"], shp.n_h, shp.d_h)
    assert_close(host(dec.u), ref_u, shp.dtype, what="u (pre-merged)")


# --------------------------------------------------------------------- the MHA path (several new tokens)
MHA_CASES = [("tiny", [5, 0], 3), ("minimind", [40, 7, 0], 6), ("v2", [150, 3], 140), ("v2", [0, 77], 300)]


@pytest.mark.parametrize("name", SMALL)
@pytest.mark.parametrize("proj", PROJ)
def test_project_q_and_materialise_kv_match_oracle(name, proj):
    shp = small_shape(name)
    W = S.draw_weights(shp)
    N = 37 if name != "tiny" else 5
    h = S.draw_new_tokens(shp, N)
    max_pos = 3000
    pos = np.random.default_rng(17).integers(0, max_pos, size=N)
    pos[0], pos[-1] = 0, max_pos - 1
    dec = decoder(shp, make_weights_dev(shp, W), N, 16, max_pos=max_pos)
    set_proj(dec, proj)
    q = torch.empty((N, shp.n_h, shp.d_h + shp.d_r), dtype=torch_dtype(shp), device="cuda")
    M.mla_project_q(dec.handle, dev(h, shp), N, dec.W["W_DQ"], dec.W["W_UQ"], dec.W["W_QR"], dev_i32(pos), q,
                    dec.ws, dec.ws.numel())
    ref_q = O.materialised_query(h, W["W_DQ"], W["W_UQ"], W["W_QR"], pos, shp.n_h, shp.d_h, shp.d_r,
                                 shp.rope_base)
    assert_close(host(q), ref_q, shp.dtype, what="q")
    rows = S.draw_latent_rows(shp, 300, sub=21)
    k_c = torch.empty((300, shp.n_h, shp.d_h), dtype=torch_dtype(shp), device="cuda")
    v_c = torch.empty_like(k_c)
    M.mla_materialise_kv(dec.handle, dev(rows, shp), 300, dec.W["W_UK"], dec.W["W_UV"], k_c, v_c)
    ref_k, ref_v = O.materialised_kv(rows, W["W_UK"], W["W_UV"], shp.n_h, shp.d_h)
    assert_close(host(k_c), ref_k, shp.dtype, what="k_C")
    assert_close(host(v_c), ref_v, shp.dtype, what="v_C")
    assert M.mla_get_device_status(dec.handle) == (M.MLA_OK, 0)


@pytest.mark.parametrize("name,ctx,n_q", MHA_CASES)
@pytest.mark.parametrize("path", ["auto", "simt"])
def test_mha_attn_matches_oracle(name, ctx, n_q, path):
    """Causal attention over stand-alone materialised inputs (unit-variance scores)."""
    shp = small_shape(name)
    B = len(ctx)
    max_len = max(ctx) + n_q + 3
    DQ = shp.d_h + shp.d_r
    q = S.draw_gaussian(shp, "spare0", (B, n_q, shp.n_h, DQ), sub=1)
    k_c = S.draw_gaussian(shp, "spare0", (B, max_len, shp.n_h, shp.d_h), sub=2)
    v_c = S.draw_gaussian(shp, "spare0", (B, max_len, shp.n_h, shp.d_h), sub=3)
    cache = S.draw_gaussian(shp, "spare0", (B, max_len, shp.D), sub=4)
    q_pos0 = np.array(ctx)
    W = {k: np.zeros(shp.weight_shape(k)) for k in S.WEIGHT_NAMES}
    dec = decoder(shp, {k: torch.zeros(1, device="cuda") for k in W}, B, max_len)
    if path == "simt":
        M.mla_set_decode_path(dec.handle, M.MLA_DECODE_SIMT)
    o = torch.empty((B, n_q, shp.n_h, shp.d_h), dtype=torch_dtype(shp), device="cuda")
    lse = torch.empty((B, n_q, shp.n_h), dtype=torch.float32, device="cuda")
    M.mla_mha_attn(dec.handle, dev(q, shp), B, n_q, dev(k_c, shp), dev(v_c, shp), dev(cache, shp), max_len,
                   dev_i32(q_pos0), o, lse)
    assert M.mla_get_device_status(dec.handle) == (M.MLA_OK, 0)
    sc = O.scale_of(shp.d_h, shp.d_r)
    got_o, got_l = host(o), lse.cpu().numpy().astype(np.float64)
    for b in range(B):
        ref_o, ref_l = O.mha_attention(q[b], k_c[b], cache[b][:, shp.d_c:], v_c[b], q_pos0[b] + np.arange(n_q), sc)
        assert_close(got_o[b], ref_o, shp.dtype, what=f"o seq {b}")
        assert np.abs(got_l[b] - ref_l).max() <= 2e-4 * max(1.0, np.abs(ref_l).max()), "lse"


@pytest.mark.parametrize("name,ctx,n_q", MHA_CASES)
def test_mha_path_end_to_end(name, ctx, n_q):
    """New tokens appended, K/V materialised, queries projected, causal MHA and
    W_O, chained on the GPU, against the oracle's prefill definition."""
    shp = small_shape(name)
    B = len(ctx)
    max_len = max(ctx) + n_q
    W = S.draw_weights(shp)
    h_ctx = [S.draw_context_h(shp, b, n) for b, n in enumerate(ctx)]
    h_new = [S.draw_gaussian(shp, "spare1", (n_q, shp.d), sub=b) for b in range(B)]
    dec = decoder(shp, make_weights_dev(shp, W), B * n_q, max_len, max_pos=max_len)
    cache = torch.zeros((B, max_len, shp.D), dtype=torch_dtype(shp), device="cuda")
    toks = np.concatenate([np.concatenate([h_ctx[b], h_new[b]]) for b in range(B)])
    seq = np.concatenate([np.full(ctx[b] + n_q, b) for b in range(B)])
    pos = np.concatenate([np.arange(ctx[b] + n_q) for b in range(B)])
    dec.append(dev(toks, shp), dev_i32(seq), dev_i32(pos), cache)
    k_c = torch.empty((B, max_len, shp.n_h, shp.d_h), dtype=torch_dtype(shp), device="cuda")
    v_c = torch.empty_like(k_c)
    M.mla_materialise_kv(dec.handle, cache, B * max_len, dec.W["W_UK"], dec.W["W_UV"], k_c, v_c)
    q = torch.empty((B, n_q, shp.n_h, shp.d_h + shp.d_r), dtype=torch_dtype(shp), device="cuda")
    qpos = np.concatenate([ctx[b] + np.arange(n_q) for b in range(B)])
    M.mla_project_q(dec.handle, dev(np.concatenate(h_new), shp), B * n_q, dec.W["W_DQ"], dec.W["W_UQ"],
                    dec.W["W_QR"], dev_i32(qpos), q, dec.ws, dec.ws.numel())
    o = torch.empty((B, n_q, shp.n_h, shp.d_h), dtype=torch_dtype(shp), device="cuda")
    lse = torch.empty((B, n_q, shp.n_h), dtype=torch.float32, device="cuda")
    M.mla_mha_attn(dec.handle, q, B, n_q, k_c, v_c, cache, max_len, dev_i32(np.array(ctx)), o, lse)
    u = torch.empty((B * n_q, shp.d), dtype=torch_dtype(shp), device="cuda")
    M.mla_project_out(dec.handle, o, B * n_q, dec.W["W_O"], u)
    assert M.mla_get_device_status(dec.handle) == (M.MLA_OK, 0)
    ref_u, ref_o, ref_l = O.prefill_materialised(h_ctx, h_new, W, shp.n_h, shp.d_h, shp.d_r, shp.rope_base,
                                                 return_parts=True)
    got_u = host(u).reshape(B, n_q, shp.d)
    got_l = lse.cpu().numpy().astype(np.float64)
    for b in range(B):
        assert_close(got_u[b], ref_u[b], shp.dtype, tol=TOL_E2E, what=f"u seq {b}")
        assert np.abs(got_l[b] - ref_l[b]).max() <= TOL_LSE_E2E_MANY[shp.dtype], "lse"


# --------------------------------------------------------------------- whole step
def end_to_end(shp, ctx_lens):
    B = len(ctx_lens)
    W = S.draw_weights(shp)
    h_ctx = [S.draw_context_h(shp, b, int(n)) for b, n in enumerate(ctx_lens)]
    h_new = S.draw_new_tokens(shp, B)
    max_len = int(max(ctx_lens)) + 1
    dec = decoder(shp, make_weights_dev(shp, W), B, max_len)
    cache = torch.zeros((B, max_len, shp.D), dtype=torch_dtype(shp), device="cuda")
    seq = np.concatenate([np.full(int(n), b) for b, n in enumerate(ctx_lens)])
    pos = np.concatenate([np.arange(int(n)) for n in ctx_lens])
    if len(seq):
        dec.append(dev(np.concatenate(h_ctx), shp), dev_i32(seq), dev_i32(pos), cache)
    # the four entry points, so that o_lat and lse stay in the decoder's buffers
    # (mla_decode_step is checked against this sequence of calls elsewhere)
    u = dec.step_calls(dev(h_new, shp), dev_i32(ctx_lens), cache, dev_i32(np.asarray(ctx_lens) + 1))
    st, bits = M.mla_get_device_status(dec.handle)
    assert st == M.MLA_OK and bits == 0
    ref_u = O.decode_materialised(h_ctx, h_new, W, shp.n_h, shp.d_h, shp.d_r, shp.rope_base)
    _, ref_o, ref_l, _, _ = O.decode_absorbed(h_ctx, h_new, W, shp.n_h, shp.d_h, shp.d_r, shp.rope_base)
    return host(u), ref_u, host(dec.o_lat), ref_o, dec.lse.cpu().numpy(), ref_l


@pytest.mark.parametrize("name,ctx", [("tiny", [128, 128]), ("minimind", [300, 0, 45, 129]),
                                      ("v2", [200, 1, 77])])
def test_decode_step_end_to_end(name, ctx):
    shp = S.workload(name)
    u, ref_u, o, ref_o, l, ref_l = end_to_end(shp, ctx)
    assert_close(o, ref_o, shp.dtype, tol=TOL_E2E, what="o_lat")
    assert_close(u, ref_u, shp.dtype, tol=TOL_E2E, what="u")
    assert np.abs(l - ref_l).max() <= TOL_LSE_E2E[shp.dtype], np.abs(l - ref_l).max()


# --------------------------------------------------------------------- full-size workloads (sampled)
FULL = ["minimind", "v2", "v2_ragged", "v2_long"]


@pytest.mark.parametrize("name", FULL)
def test_decode_attn_full_size_sampled(name):
    """The workload's full batch and context, in the launch configuration the
    benchmark times; the oracle checks three sampled sequences (shortest,
    longest, one more)."""
    shp = S.workload(name)
    ctx = S.draw_context_lengths(shp)
    seqlens = ctx + 1
    B, max_len = len(seqlens), int(seqlens.max())
    g = torch.Generator(device="cuda")
    g.manual_seed(shp.seed)
    cache = torch.randn((B, max_len, shp.D), generator=g, device="cuda", dtype=torch.float32).to(torch_dtype(shp))
    q = S.draw_absorbed_queries(shp, B)
    dec = decoder(shp, {k: torch.zeros(1, device="cuda") for k in S.WEIGHT_NAMES}, B, max_len)
    M.mla_decode_attn(dec.handle, dev(q, shp), cache, B, max_len, dev_i32(seqlens), dec.o_lat, dec.lse, dec.ws,
                      dec.ws.numel())
    st, bits = M.mla_get_device_status(dec.handle)
    assert st == M.MLA_OK and bits == 0
    picks = sorted({int(np.argmin(seqlens)), int(np.argmax(seqlens)), B // 2})
    sc = O.scale_of(shp.d_h, shp.d_r)
    for b in picks:
        rows = host(cache[b, :seqlens[b]])
        ref_o, ref_l = O.latent_attention(q[b], rows, shp.d_c, sc)
        assert_close(host(dec.o_lat[b]), ref_o, shp.dtype, what=f"o_lat[{b}]")
        assert np.abs(dec.lse[b].cpu().numpy() - ref_l).max() <= 2e-4 * max(1, np.abs(ref_l).max())


@pytest.mark.gpu
def test_captured_step_matches_eager():
    """MLADecoder.capture/replay: the step recorded as a CUDA graph gives the
    same cache row and output as the eager step (same kernels, same inputs)."""
    shp = S.workload("v2")
    B, L = 4, 300
    W = S.draw_weights(shp)
    dec = decoder(shp, make_weights_dev(shp, W), B, L, max_pos=L)
    rng = np.random.default_rng(11)
    cache0 = dev(rng.standard_normal((B, L, shp.D)), shp)
    h = dev(S.draw_context_h(shp, 1, B), shp)
    pos = dev_i32(rng.integers(0, L - 1, size=B))
    seqlens = dev_i32(host(pos) + 1)
    cache_e = cache0.clone()
    u_e = dec.step(h, pos, cache_e, seqlens).clone()
    cache_g = cache0.clone()
    dec.capture(cache_g)
    dec.h_in.copy_(h)
    dec.pos_in.copy_(pos)
    dec.seqlens_in.copy_(seqlens)
    u_g = dec.replay().clone()
    torch.cuda.synchronize()
    assert torch.equal(u_g, u_e)
    assert torch.equal(cache_g, cache_e)
    st, bits = M.mla_get_device_status(dec.handle)
    assert st == M.MLA_OK and bits == 0
    dec.close()


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["minimind", "v2"])
def test_step_call_matches_four_calls(name):
    """mla_decode_step (S1 and c_Q in one launch where the tensor-core kernel
    takes both; MiniMind's W_UK^T falls back) writes the same cache rows and u
    as the four entry points called in turn. The fused launch may cut K into
    other split-K pieces than the separate S1 and c_Q launches (one choice for
    all its tiles), so its fp32 sums can associate differently: a stored
    element then agrees to one bf16 rounding step, u to the end-to-end
    tolerance."""
    shp = S.workload(name)
    B, L = 6, 400
    W = S.draw_weights(shp)
    dec = decoder(shp, make_weights_dev(shp, W), B, L, max_pos=L)
    rng = np.random.default_rng(12)
    cache0 = dev(rng.standard_normal((B, L, shp.D)), shp)
    h = dev(S.draw_context_h(shp, 2, B), shp)
    pos = dev_i32(rng.integers(0, L - 1, size=B))
    seqlens = dev_i32(host(pos) + 1)
    cache_a = cache0.clone()
    u_a = dec.step_calls(h, pos, cache_a, seqlens).clone()
    cache_b = cache0.clone()
    u_b = dec.step(h, pos, cache_b, seqlens).clone()
    torch.cuda.synchronize()
    a, b = host(cache_a), host(cache_b)
    step = 2.0 ** -7 if shp.dtype == "bf16" else 2.0 ** -23
    assert (np.abs(a - b) <= step * np.maximum(np.abs(a), np.abs(b))).all()
    assert (a != b).mean() < 0.02
    assert_close(host(u_b), host(u_a), shp.dtype, tol=TOL_E2E, what="u, fused step vs four calls")
    st, bits = M.mla_get_device_status(dec.handle)
    assert st == M.MLA_OK and bits == 0
    dec.close()


# --------------------------------------------------------------------- bounded waits
@pytest.mark.parametrize("name", ["minimind", "v2"])
def test_decode_attn_wait_timeout_then_recovers(name):
    """Failure detection without a GPU fault: with a short wait limit and the
    test hook that withholds one internal arrival, the tensor-core attention
    kernel gives up, flags MLA_DEV_TIMEOUT and returns; the next call on the
    same handle and context is correct again."""
    shp = S.workload(name)
    max_len = 300
    seqlens = np.array([300, 129, 1, 77])
    B = len(seqlens)
    q = S.draw_absorbed_queries(shp, B)
    rows = [S.draw_latent_rows(shp, int(n), sub=80 + b) for b, n in enumerate(seqlens)]
    cache = np.zeros((B, max_len, shp.D))
    for b, r in enumerate(rows):
        cache[b, :len(r)] = r
    dec = decoder(shp, {k: torch.zeros(1, device="cuda") for k in S.WEIGHT_NAMES}, B, max_len)
    assert M.mla_get_decode_path(dec.handle) == M.MLA_DECODE_TCGEN05
    qd, cd, sl = dev(q, shp), dev(cache, shp), dev_i32(seqlens)
    M.mla_set_wait_limit(dec.handle, 20_000_000)      # ~10 ms of SM clocks
    M.mla_set_fault_injection(dec.handle, 1)
    M.mla_decode_attn(dec.handle, qd, cd, B, max_len, sl, dec.o_lat, dec.lse, dec.ws, dec.ws.numel())
    st, bits = M.mla_get_device_status(dec.handle)
    assert st == M.MLA_ERR_TIMEOUT and bits & M.MLA_DEV_TIMEOUT
    M.mla_set_fault_injection(dec.handle, 0)
    M.mla_set_wait_limit(dec.handle, 0)
    dec.o_lat.zero_()
    M.mla_decode_attn(dec.handle, qd, cd, B, max_len, sl, dec.o_lat, dec.lse, dec.ws, dec.ws.numel())
    st, bits = M.mla_get_device_status(dec.handle)
    assert st == M.MLA_OK and bits == 0
    ref_o, ref_l = oracle_decode(shp, q, rows, seqlens)
    assert_close(host(dec.o_lat), ref_o, shp.dtype, what="o_lat after recovery")
    assert np.abs(dec.lse.cpu().numpy() - ref_l).max() <= 2e-4 * max(1, np.abs(ref_l).max())
    dec.close()


def test_decode_attn_few_head_kernel_agrees_with_cuda_core():
    """The MiniMind-shaped layer takes the few-head tensor-core kernel by
    default; it agrees with the CUDA-core kernel on the same inputs."""
    shp = S.workload("minimind")
    max_len = 700
    seqlens = np.array([700, 129, 1, 640, 0, 333])
    q = S.draw_absorbed_queries(shp, len(seqlens))
    rows = [S.draw_latent_rows(shp, int(n), sub=b) for b, n in enumerate(seqlens)]
    a = run_decode(shp, q, rows, seqlens, max_len, path=M.MLA_DECODE_SIMT)
    b = run_decode(shp, q, rows, seqlens, max_len, path=M.MLA_DECODE_AUTO)
    assert M.mla_get_decode_path(b[4].handle) == M.MLA_DECODE_TCGEN05
    nz = seqlens > 0
    assert_close(b[0][nz], a[0][nz], "bf16")
    assert np.all(b[0][~nz] == 0) and np.all(np.isneginf(b[1][~nz]))


# --------------------------------------------------------------------- the benchmarked step at full size
def test_decode_step_full_size_v2_sampled():
    """mla_decode_step at the benchmark's size (V2 layer, batch 64, 4096 cached
    tokens per sequence appended through mla_append_cache, one new token at
    position 4096): the new cache rows and u of three sampled sequences match
    the fp64 materialised definition (per-head k_C = W_UK c_KV, v_C = W_UV c_KV,
    two-pass softmax, W_O)."""
    shp = S.workload("v2")
    B, ctx = shp.batch, shp.ctx
    max_len = ctx + 1
    W = S.draw_weights(shp)
    dec = decoder(shp, make_weights_dev(shp, W), B, max_len, max_pos=max_len)
    cache = torch.zeros((B, max_len, shp.D), dtype=torch.bfloat16, device="cuda")
    per = 8
    for b0 in range(0, B, per):
        bs = list(range(b0, b0 + per))
        x = torch.cat([S.context_h_device(shp, b, ctx, "cuda") for b in bs], 0).contiguous()
        seq = dev_i32(np.repeat(bs, ctx))
        pos = dev_i32(np.tile(np.arange(ctx), per))
        dec.append(x, seq, pos, cache)
    h_new = S.draw_new_tokens(shp, B)
    pos = np.full(B, ctx)
    u = dec.step(dev(h_new, shp), dev_i32(pos), cache, dev_i32(pos + 1))
    st, bits = M.mla_get_device_status(dec.handle)
    assert st == M.MLA_OK and bits == 0
    got_u = host(u)
    for b in (0, 31, 63):
        h_ctx = host(S.context_h_device(shp, b, ctx, "cuda"))
        ref_u = O.decode_materialised([h_ctx], h_new[b:b + 1], W, shp.n_h, shp.d_h, shp.d_r, shp.rope_base)
        assert_close(got_u[b:b + 1], ref_u, shp.dtype, tol=TOL_E2E, what=f"u[{b}]")
        ref_row = O.cache_rows(h_new[b:b + 1], W["W_DKV"], W["W_KR"], [ctx], shp.rope_base)
        assert_close(host(cache[b, ctx:ctx + 1]), ref_row, shp.dtype, what=f"new cache row [{b}]")
    dec.close()


# --------------------------------------------------------------------- the kv_norm variant
@pytest.mark.parametrize("name", SMALL)
@pytest.mark.parametrize("proj", PROJ)
def test_append_kv_norm_matches_oracle(name, proj):
    """mla_set_kv_norm: appended rows carry the RMS-normalised latent (MiniMind
    page §9, kv_norm on kv_latent) and the unchanged RoPE key; rows not
    appended stay untouched."""
    shp = small_shape(name)
    W = S.draw_weights(shp)
    rng = np.random.default_rng(31)
    g = S.to_dtype(rng.uniform(0.5, 1.5, size=shp.d_c), shp.dtype)
    B, L, n = 3, 200, 300
    flat = rng.choice(B * L, size=n, replace=False)
    seq, pos = flat // L, flat % L
    x = S.draw_context_h(shp, 3, n)
    dec = decoder(shp, make_weights_dev(shp, W), B, L)
    set_proj(dec, proj)
    g_dev = dev(g, shp)   # the library keeps the pointer: the tensor must outlive the appends
    M.mla_set_kv_norm(dec.handle, g_dev, 1e-5)
    cache = torch.full((B, L, shp.D), float("nan"), dtype=torch_dtype(shp), device="cuda")
    dec.append(dev(x, shp), dev_i32(seq), dev_i32(pos), cache)
    st, bits = M.mla_get_device_status(dec.handle)
    assert st == M.MLA_OK and bits == 0
    got = host(cache)
    ref = O.cache_rows(x, W["W_DKV"], W["W_KR"], pos, shp.rope_base, kv_norm_weight=g, kv_norm_eps=1e-5)
    assert_close(got[seq, pos], ref, shp.dtype, what="normalised cache rows")
    untouched = np.ones((B, L), bool)
    untouched[seq, pos] = False
    assert np.isnan(got[untouched]).all()
    dec.close()


@pytest.mark.parametrize("name,ctx", [("tiny", [100, 64]), ("minimind", [200, 33, 1]), ("v2", [150, 7])])
def test_decode_step_kv_norm_end_to_end(name, ctx):
    """The whole step with kv_norm on (context appended through mla_append_cache,
    the new token through mla_decode_step) against the materialised definition
    with K and V expanded from the normalised latent."""
    shp = S.workload(name)
    W = S.draw_weights(shp)
    g = S.to_dtype(np.random.default_rng(32).uniform(0.5, 1.5, size=shp.d_c), shp.dtype)
    B = len(ctx)
    h_ctx = [S.draw_context_h(shp, b, int(n)) for b, n in enumerate(ctx)]
    h_new = S.draw_new_tokens(shp, B)
    max_len = int(max(ctx)) + 1
    dec = decoder(shp, make_weights_dev(shp, W), B, max_len)
    g_dev = dev(g, shp)   # the library keeps the pointer: the tensor must outlive the step
    M.mla_set_kv_norm(dec.handle, g_dev, 1e-5)
    cache = torch.zeros((B, max_len, shp.D), dtype=torch_dtype(shp), device="cuda")
    seq = np.concatenate([np.full(int(n), b) for b, n in enumerate(ctx)])
    pos = np.concatenate([np.arange(int(n)) for n in ctx])
    dec.append(dev(np.concatenate(h_ctx), shp), dev_i32(seq), dev_i32(pos), cache)
    u = dec.step(dev(h_new, shp), dev_i32(ctx), cache, dev_i32(np.asarray(ctx) + 1))
    st, bits = M.mla_get_device_status(dec.handle)
    assert st == M.MLA_OK and bits == 0
    ref_u = O.decode_materialised(h_ctx, h_new, W, shp.n_h, shp.d_h, shp.d_r, shp.rope_base, kv_norm_weight=g,
                                  kv_norm_eps=1e-5)
    assert_close(host(u), ref_u, shp.dtype, tol=TOL_E2E, what="u with kv_norm")
    dec.close()
