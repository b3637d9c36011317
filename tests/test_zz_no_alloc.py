"""mla_decode_attn_noalloc — the decode attention entry point for callers that
cannot allocate device memory (for instance an engine whose own pool owns all
device memory, or a loop that cannot afford cudaMalloc's implicit device
synchronisation). It takes no workspace and keeps its scratch in the library's
fixed device array.

Checked through the C ABI against mla_decode_attn (the entry point that takes
caller workspace) on the same inputs, within the parity tolerance used for the
decode tests, on two calls in a row with different inputs, so the second call
runs on the scratch contents the first one left behind. Collected last so that
a run stopping at the first failure has already run every other test."""
import numpy as np
import pytest

import mla_synth as S
from gpu_helpers import assert_close, dev, dev_i32, host, decoder

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)
import head_latent_attention_24_b300 as M  # noqa: E402


def _case(shp, seqlens, max_len, sub):
    B = len(seqlens)
    q = S.draw_absorbed_queries(shp, B, sub=sub)
    cache = np.zeros((B, max_len, shp.D))
    for b, n in enumerate(seqlens):
        cache[b, :n] = S.draw_latent_rows(shp, int(n), sub=100 * sub + b)
    return dev(q, shp), dev(cache, shp), dev_i32(seqlens)


def _with_workspace(shp, q, cache, sl, B, max_len):
    dec = decoder(shp, {k: torch.zeros(1, device="cuda") for k in S.WEIGHT_NAMES}, B, max_len)
    M.mla_set_decode_path(dec.handle, M.MLA_DECODE_SIMT)
    M.mla_decode_attn(dec.handle, q, cache, B, max_len, sl, dec.o_lat, dec.lse, dec.ws, dec.ws.numel())
    torch.cuda.synchronize()
    return host(dec.o_lat), dec.lse.double().cpu().numpy()


def _no_alloc(shp, q, cache, sl, B, max_len):
    o = torch.full((B, shp.n_h, shp.d_c), float("nan"), dtype=q.dtype, device="cuda")
    lse = torch.full((B, shp.n_h), float("nan"), dtype=torch.float32, device="cuda")
    M.mla_decode_attn_noalloc(shp.n_h, shp.d_h, shp.d_c, shp.d_r, M.MLA_BF16 if shp.dtype == "bf16" else M.MLA_F32,
                              q, cache, B, max_len, sl, o, lse)
    torch.cuda.synchronize()
    return host(o), lse.double().cpu().numpy()


@pytest.mark.parametrize("name,calls", [
    ("minimind", [(np.array([700, 1, 0, 333, 64, 65, 512, 699]), 700),
                  (np.array([5, 640, 77, 700, 300, 2]), 700)]),
    ("v2", [(np.array([300, 129, 1]), 300), (np.array([64, 0, 250, 300]), 300)]),
    ("tiny", [(np.array([129, 129]), 129), (np.array([17, 128]), 129)]),
])
def test_no_alloc_matches_workspace_entry_point_on_two_calls(name, calls):
    shp = S.workload(name)
    for i, (seqlens, max_len) in enumerate(calls):
        B = len(seqlens)
        q, cache, sl = _case(shp, seqlens, max_len, sub=i + 1)
        ref_o, ref_l = _with_workspace(shp, q, cache, sl, B, max_len)
        got_o, got_l = _no_alloc(shp, q, cache, sl, B, max_len)
        nz = seqlens > 0
        assert_close(got_o[nz], ref_o[nz], shp.dtype, what=f"call {i + 1} o_lat")
        assert np.all(got_o[~nz] == 0) and np.all(np.isneginf(got_l[~nz]))
        assert np.abs(got_l[nz] - ref_l[nz]).max() <= 2e-4 * max(1.0, np.abs(ref_l[nz]).max())


def test_no_alloc_rejects_requests_beyond_its_scratch():
    shp = S.workload("v2")
    B, max_len = 64, 8
    q = torch.zeros((B, shp.n_h, shp.D), dtype=torch.bfloat16, device="cuda")
    cache = torch.zeros((B, max_len, shp.D), dtype=torch.bfloat16, device="cuda")
    sl = dev_i32(np.full(B, max_len))
    o = torch.zeros((B, shp.n_h, shp.d_c), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((B, shp.n_h), dtype=torch.float32, device="cuda")
    with pytest.raises(M.MLAError) as e:
        M.mla_decode_attn_noalloc(shp.n_h, shp.d_h, shp.d_c, shp.d_r, M.MLA_BF16, q, cache, B, max_len, sl, o, lse)
    assert e.value.status == M.MLA_ERR_WORKSPACE
