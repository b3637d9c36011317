"""Python binding of libmla.so, the sm_103a MLA decode library.

Argument marshalling only: every function below passes device pointers, sizes
and the current CUDA stream to the C entry point of the same name
(include/mla.h) and raises MLAError on a non-zero status. PyTorch supplies the
device memory and streams; all arithmetic runs in the library's kernels.
Importing this package fails if libmla.so has not been built
(``python head_latent_attention_24_b300/build.py``) — there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmla.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with `python head_latent_attention_24_b300/build.py`")

_lib = ctypes.CDLL(LIB_PATH)

# ----------------------------------------------------------------- constants
MLA_OK = 0
MLA_ERR_INVALID_ARG = -1
MLA_ERR_UNSUPPORTED = -2
MLA_ERR_CUDA = -3
MLA_ERR_DEVICE = -4
MLA_ERR_TIMEOUT = -5
MLA_ERR_WORKSPACE = -6
MLA_F32 = 0
MLA_BF16 = 1
MLA_DEV_SEQLEN_RANGE = 0x1
MLA_DEV_POS_RANGE = 0x2
MLA_DEV_SEQ_RANGE = 0x4
MLA_DEV_QPOS_RANGE = 0x8
MLA_DEV_TIMEOUT = 0x10
MLA_DECODE_AUTO = 0
MLA_DECODE_SIMT = 1
MLA_DECODE_TCGEN05 = 2
MLA_PROJ_AUTO = 0
MLA_PROJ_SIMT = 1
MLA_PROJ_TCGEN05 = 2


class mla_config_t(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int32), ("n_h", ctypes.c_int32), ("d_h", ctypes.c_int32),
                ("d_c", ctypes.c_int32), ("d_r", ctypes.c_int32), ("d_cq", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("max_pos", ctypes.c_int32), ("rope_base", ctypes.c_double)]


class MLAError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {mla_status_string(status)} ({status})")


_P = ctypes.c_void_p
_I = ctypes.c_int32
_S = ctypes.c_size_t


def _sig(name, args, res=ctypes.c_int32):
    f = getattr(_lib, name)
    f.argtypes = args
    f.restype = res
    return f


_c = {
    "mla_abi_version": _sig("mla_abi_version", []),
    "mla_status_string": _sig("mla_status_string", [_I], ctypes.c_char_p),
    "mla_create": _sig("mla_create", [ctypes.POINTER(mla_config_t), ctypes.POINTER(_P)]),
    "mla_destroy": _sig("mla_destroy", [_P]),
    "mla_append_cache": _sig("mla_append_cache", [_P, _P, _I, _P, _P, _P, _P, _P, _I, _I, _P]),
    "mla_absorb_q_workspace_size": _sig("mla_absorb_q_workspace_size", [_P, _I, ctypes.POINTER(_S)]),
    "mla_absorb_q": _sig("mla_absorb_q", [_P, _P, _I, _P, _P, _P, _P, _P, _P, _P, _S, _P]),
    "mla_decode_workspace_size": _sig("mla_decode_workspace_size", [_P, _I, _I, ctypes.POINTER(_S)]),
    "mla_decode_attn": _sig("mla_decode_attn", [_P, _P, _P, _I, _I, _P, _P, _P, _P, _S, _P]),
    "mla_decode_attn_noalloc": _sig("mla_decode_attn_noalloc", [_I, _I, _I, _I, _I, _P, _P, _I, _I, _P, _P, _P, _P]),
    "mla_out_proj_workspace_size": _sig("mla_out_proj_workspace_size", [_P, _I, ctypes.POINTER(_S)]),
    "mla_out_proj": _sig("mla_out_proj", [_P, _P, _I, _P, _P, _P, _P, _S, _P]),
    "mla_decode_step_workspace_size": _sig("mla_decode_step_workspace_size", [_P, _I, _I, ctypes.POINTER(_S)]),
    "mla_decode_step": _sig("mla_decode_step", [_P, _P, _I] + [_P] * 8 + [_P, _P, _P, _I, _P, _P, _S, _P]),
    "mla_get_device_status": _sig("mla_get_device_status", [_P, _P, ctypes.POINTER(_I)]),
    "mla_set_decode_path": _sig("mla_set_decode_path", [_P, _I]),
    "mla_set_decode_chunks": _sig("mla_set_decode_chunks", [_P, _I]),
    "mla_get_decode_path": _sig("mla_get_decode_path", [_P, ctypes.POINTER(_I)]),
    "mla_set_proj_path": _sig("mla_set_proj_path", [_P, _I]),
    "mla_last_launch_count": _sig("mla_last_launch_count", [_P, ctypes.POINTER(_I)]),
    "mla_set_wait_limit": _sig("mla_set_wait_limit", [_P, ctypes.c_int64]),
    "mla_set_kv_norm": _sig("mla_set_kv_norm", [_P, _P, ctypes.c_float]),
    "mla_set_fault_injection": _sig("mla_set_fault_injection", [_P, _I]),
    "mla_premerge_query_weights": _sig("mla_premerge_query_weights", [_P, _P, _P, _P, _P]),
    "mla_premerge_output_weights": _sig("mla_premerge_output_weights", [_P, _P, _P, _P, _P]),
    "mla_absorb_q_premerged": _sig("mla_absorb_q_premerged", [_P, _P, _I, _P, _P, _P, _P, _P, _P, _S, _P]),
    "mla_out_proj_premerged": _sig("mla_out_proj_premerged", [_P, _P, _I, _P, _P, _P]),
    "mla_project_q": _sig("mla_project_q", [_P, _P, _I, _P, _P, _P, _P, _P, _P, _S, _P]),
    "mla_materialise_kv": _sig("mla_materialise_kv", [_P, _P, _I, _P, _P, _P, _P, _P]),
    "mla_mha_attn": _sig("mla_mha_attn", [_P, _P, _I, _I, _P, _P, _P, _I, _P, _P, _P, _P]),
    "mla_project_out": _sig("mla_project_out", [_P, _P, _I, _P, _P, _P]),
}


def _check(st: int, what: str):
    if st != MLA_OK:
        raise MLAError(st, what)


def _ptr(t):
    """Device pointer of a tensor (None -> NULL). Tensors must be dense."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ----------------------------------------------------------------- entry points
def mla_abi_version() -> int:
    return _c["mla_abi_version"]()


def mla_status_string(status: int) -> str:
    return _c["mla_status_string"](status).decode()


def mla_create(d, n_h, d_h, d_c, d_r, d_cq, dtype, max_pos, rope_base=10000.0):
    cfg = mla_config_t(d, n_h, d_h, d_c, d_r, d_cq, dtype, max_pos, rope_base)
    h = _P()
    _check(_c["mla_create"](ctypes.byref(cfg), ctypes.byref(h)), "mla_create")
    return h


def mla_destroy(handle):
    _check(_c["mla_destroy"](handle), "mla_destroy")


def mla_append_cache(handle, x, n_tokens, W_DKV, W_KR, tok_seq, tok_pos, cache, batch, max_len, stream=None):
    _check(_c["mla_append_cache"](handle, _ptr(x), n_tokens, _ptr(W_DKV), _ptr(W_KR), _ptr(tok_seq),
                                  _ptr(tok_pos), _ptr(cache), batch, max_len, _stream(stream)),
           "mla_append_cache")


def mla_absorb_q_workspace_size(handle, batch) -> int:
    n = _S()
    _check(_c["mla_absorb_q_workspace_size"](handle, batch, ctypes.byref(n)), "mla_absorb_q_workspace_size")
    return n.value


def mla_absorb_q(handle, x, batch, W_DQ, W_UQ, W_QR, W_UK, pos, q_abs, ws, ws_bytes, stream=None):
    _check(_c["mla_absorb_q"](handle, _ptr(x), batch, _ptr(W_DQ), _ptr(W_UQ), _ptr(W_QR), _ptr(W_UK),
                              _ptr(pos), _ptr(q_abs), _ptr(ws), ws_bytes, _stream(stream)), "mla_absorb_q")


def mla_decode_workspace_size(handle, batch, max_len) -> int:
    n = _S()
    _check(_c["mla_decode_workspace_size"](handle, batch, max_len, ctypes.byref(n)), "mla_decode_workspace_size")
    return n.value


def mla_decode_attn(handle, q_abs, cache, batch, max_len, seqlens, o_lat, lse, ws, ws_bytes, stream=None):
    _check(_c["mla_decode_attn"](handle, _ptr(q_abs), _ptr(cache), batch, max_len, _ptr(seqlens), _ptr(o_lat),
                                 _ptr(lse), _ptr(ws), ws_bytes, _stream(stream)), "mla_decode_attn")


def mla_decode_attn_noalloc(n_h, d_h, d_c, d_r, dtype, q_abs, cache, batch, max_len, seqlens, o_lat, lse,
                            stream=None):
    """Decode attention with no workspace argument and no allocation (scratch is
    the library's own fixed device array; see include/mla.h)."""
    _check(_c["mla_decode_attn_noalloc"](n_h, d_h, d_c, d_r, dtype, _ptr(q_abs), _ptr(cache), batch, max_len,
                                         _ptr(seqlens), _ptr(o_lat), _ptr(lse), _stream(stream)),
           "mla_decode_attn_noalloc")


def mla_out_proj_workspace_size(handle, batch) -> int:
    n = _S()
    _check(_c["mla_out_proj_workspace_size"](handle, batch, ctypes.byref(n)), "mla_out_proj_workspace_size")
    return n.value


def mla_out_proj(handle, o_lat, batch, W_UV, W_O, u, ws, ws_bytes, stream=None):
    _check(_c["mla_out_proj"](handle, _ptr(o_lat), batch, _ptr(W_UV), _ptr(W_O), _ptr(u), _ptr(ws), ws_bytes,
                              _stream(stream)), "mla_out_proj")


def mla_premerge_query_weights(handle, W_UQ, W_UK, W_QK, stream=None):
    """W_QK [n_h, d_c, d_cq] = W_UK_i^T W_UQ_i per head (see include/mla.h)."""
    _check(_c["mla_premerge_query_weights"](handle, _ptr(W_UQ), _ptr(W_UK), _ptr(W_QK), _stream(stream)),
           "mla_premerge_query_weights")


def mla_premerge_output_weights(handle, W_UV, W_O, W_OUV, stream=None):
    """W_OUV [d, n_h * d_c], column block i = W_O_i W_UV_i (see include/mla.h)."""
    _check(_c["mla_premerge_output_weights"](handle, _ptr(W_UV), _ptr(W_O), _ptr(W_OUV), _stream(stream)),
           "mla_premerge_output_weights")


def mla_absorb_q_premerged(handle, x, batch, W_DQ, W_QK, W_QR, pos, q_abs, ws, ws_bytes, stream=None):
    _check(_c["mla_absorb_q_premerged"](handle, _ptr(x), batch, _ptr(W_DQ), _ptr(W_QK), _ptr(W_QR), _ptr(pos),
                                        _ptr(q_abs), _ptr(ws), ws_bytes, _stream(stream)), "mla_absorb_q_premerged")


def mla_out_proj_premerged(handle, o_lat, batch, W_OUV, u, stream=None):
    _check(_c["mla_out_proj_premerged"](handle, _ptr(o_lat), batch, _ptr(W_OUV), _ptr(u), _stream(stream)),
           "mla_out_proj_premerged")


def mla_project_q(handle, x, n_tokens, W_DQ, W_UQ, W_QR, pos, q, ws, ws_bytes, stream=None):
    _check(_c["mla_project_q"](handle, _ptr(x), n_tokens, _ptr(W_DQ), _ptr(W_UQ), _ptr(W_QR), _ptr(pos), _ptr(q),
                               _ptr(ws), ws_bytes, _stream(stream)), "mla_project_q")


def mla_materialise_kv(handle, rows, n_rows, W_UK, W_UV, k_c, v_c, stream=None):
    _check(_c["mla_materialise_kv"](handle, _ptr(rows), n_rows, _ptr(W_UK), _ptr(W_UV), _ptr(k_c), _ptr(v_c),
                                    _stream(stream)), "mla_materialise_kv")


def mla_mha_attn(handle, q, batch, n_q, k_c, v_c, cache, max_len, q_pos0, o, lse, stream=None):
    _check(_c["mla_mha_attn"](handle, _ptr(q), batch, n_q, _ptr(k_c), _ptr(v_c), _ptr(cache), max_len, _ptr(q_pos0),
                              _ptr(o), _ptr(lse), _stream(stream)), "mla_mha_attn")


def mla_project_out(handle, o, n_tokens, W_O, u, stream=None):
    _check(_c["mla_project_out"](handle, _ptr(o), n_tokens, _ptr(W_O), _ptr(u), _stream(stream)), "mla_project_out")


def mla_decode_step_workspace_size(handle, batch, max_len) -> int:
    n = _S()
    _check(_c["mla_decode_step_workspace_size"](handle, batch, max_len, ctypes.byref(n)),
           "mla_decode_step_workspace_size")
    return n.value


def mla_decode_step(handle, x, batch, W_DKV, W_KR, W_DQ, W_UQ, W_QR, W_UK, W_UV, W_O, pos, seqlens, cache,
                    max_len, u, ws, ws_bytes, stream=None):
    _check(_c["mla_decode_step"](handle, _ptr(x), batch, _ptr(W_DKV), _ptr(W_KR), _ptr(W_DQ), _ptr(W_UQ),
                                 _ptr(W_QR), _ptr(W_UK), _ptr(W_UV), _ptr(W_O), _ptr(pos), _ptr(seqlens),
                                 _ptr(cache), max_len, _ptr(u), _ptr(ws), ws_bytes, _stream(stream)),
           "mla_decode_step")


def mla_get_device_status(handle, stream=None):
    """Returns (status, bits); does not raise on device-side flags."""
    bits = _I()
    st = _c["mla_get_device_status"](handle, _stream(stream), ctypes.byref(bits))
    if st == MLA_ERR_CUDA or st == MLA_ERR_INVALID_ARG:
        raise MLAError(st, "mla_get_device_status")
    return st, bits.value


def mla_set_decode_path(handle, path):
    _check(_c["mla_set_decode_path"](handle, path), "mla_set_decode_path")


def mla_set_decode_chunks(handle, chunks):
    _check(_c["mla_set_decode_chunks"](handle, chunks), "mla_set_decode_chunks")


def mla_get_decode_path(handle) -> int:
    p = _I()
    _check(_c["mla_get_decode_path"](handle, ctypes.byref(p)), "mla_get_decode_path")
    return p.value


def mla_set_proj_path(handle, path):
    _check(_c["mla_set_proj_path"](handle, path), "mla_set_proj_path")


def mla_set_kv_norm(handle, weight, eps=1e-5):
    """weight: device tensor [d_c] in the handle's dtype, or None to turn the norm off."""
    _check(_c["mla_set_kv_norm"](handle, _ptr(weight), eps), "mla_set_kv_norm")


def mla_set_wait_limit(handle, cycles):
    _check(_c["mla_set_wait_limit"](handle, cycles), "mla_set_wait_limit")


def mla_set_fault_injection(handle, mode):
    _check(_c["mla_set_fault_injection"](handle, mode), "mla_set_fault_injection")


def mla_last_launch_count(handle) -> int:
    n = _I()
    _check(_c["mla_last_launch_count"](handle, ctypes.byref(n)), "mla_last_launch_count")
    return n.value


# ----------------------------------------------------------------- convenience
@dataclass
class LayerShape:
    d: int
    n_h: int
    d_h: int
    d_c: int
    d_r: int
    d_cq: int
    dtype: str = "bf16"
    rope_base: float = 10000.0

    @property
    def D(self):
        return self.d_c + self.d_r


class MLADecoder:
    """One MLA layer on one GPU: a handle, the layer's weights (device tensors,
    [out, in]) and workspaces sized for a batch. ``step`` runs S1..S5 through
    the four entry points on the current stream."""

    WEIGHTS = ("W_DKV", "W_KR", "W_DQ", "W_UQ", "W_QR", "W_UK", "W_UV", "W_O")

    def __init__(self, shape: LayerShape, weights: dict, batch: int, max_len: int, max_pos: int | None = None):
        import torch
        self.shape = shape
        self.batch = batch
        self.max_len = max_len
        self.torch_dtype = torch.bfloat16 if shape.dtype == "bf16" else torch.float32
        self.handle = mla_create(shape.d, shape.n_h, shape.d_h, shape.d_c, shape.d_r, shape.d_cq,
                                 MLA_BF16 if shape.dtype == "bf16" else MLA_F32,
                                 max_pos if max_pos is not None else max_len, shape.rope_base)
        self.W = {k: weights[k] for k in self.WEIGHTS}
        dev = next(iter(self.W.values())).device
        ws = max(mla_absorb_q_workspace_size(self.handle, batch),
                 mla_decode_workspace_size(self.handle, batch, max_len),
                 mla_out_proj_workspace_size(self.handle, batch),
                 mla_decode_step_workspace_size(self.handle, batch, max_len))
        self.ws = torch.empty(ws, dtype=torch.uint8, device=dev)
        self.q_abs = torch.empty((batch, shape.n_h, shape.D), dtype=self.torch_dtype, device=dev)
        self.o_lat = torch.empty((batch, shape.n_h, shape.d_c), dtype=self.torch_dtype, device=dev)
        self.lse = torch.empty((batch, shape.n_h), dtype=torch.float32, device=dev)
        self.u = torch.empty((batch, shape.d), dtype=self.torch_dtype, device=dev)
        self.tok_seq = torch.arange(batch, dtype=torch.int32, device=dev)
        self.launches = 0

    def close(self):
        if self.handle is not None:
            mla_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def append(self, x, tok_seq, tok_pos, cache, stream=None):
        mla_append_cache(self.handle, x, x.shape[0], self.W["W_DKV"], self.W["W_KR"], tok_seq, tok_pos, cache,
                         cache.shape[0], cache.shape[1], stream)
        return mla_last_launch_count(self.handle)

    def step(self, h_new, pos, cache, seqlens, stream=None):
        """One decode step for `batch` sequences: h_new [B, d] at positions
        pos [B] (int32, device); cache [B, max_len, D]; seqlens [B] = pos + 1.
        One library call (mla_decode_step). Returns u [B, d] (the decoder's
        buffer)."""
        B = self.batch
        mla_decode_step(self.handle, h_new, B, self.W["W_DKV"], self.W["W_KR"], self.W["W_DQ"], self.W["W_UQ"],
                        self.W["W_QR"], self.W["W_UK"], self.W["W_UV"], self.W["W_O"], pos, seqlens, cache,
                        self.max_len, self.u, self.ws, self.ws.numel(), stream)
        self.launches = mla_last_launch_count(self.handle)
        return self.u

    def step_calls(self, h_new, pos, cache, seqlens, stream=None):
        """The same step through the four entry points (append, absorb,
        attention, output projection), with q_abs, o_lat and lse kept in the
        decoder's buffers. Returns u [B, d]."""
        B = self.batch
        n = 0
        mla_append_cache(self.handle, h_new, B, self.W["W_DKV"], self.W["W_KR"], self.tok_seq, pos, cache, B,
                         self.max_len, stream)
        n += mla_last_launch_count(self.handle)
        mla_absorb_q(self.handle, h_new, B, self.W["W_DQ"], self.W["W_UQ"], self.W["W_QR"], self.W["W_UK"], pos,
                     self.q_abs, self.ws, self.ws.numel(), stream)
        n += mla_last_launch_count(self.handle)
        mla_decode_attn(self.handle, self.q_abs, cache, B, self.max_len, seqlens, self.o_lat, self.lse, self.ws,
                        self.ws.numel(), stream)
        n += mla_last_launch_count(self.handle)
        mla_out_proj(self.handle, self.o_lat, B, self.W["W_UV"], self.W["W_O"], self.u, self.ws, self.ws.numel(),
                     stream)
        n += mla_last_launch_count(self.handle)
        self.launches = n
        return self.u

    def capture(self, cache):
        """Record one decode step as a CUDA graph: the step reads its inputs
        from the decoder's buffers h_in [B, d], pos_in [B] and seqlens_in [B]
        (copy each step's values into them) and works on `cache`; replay()
        then runs the whole step with one launch from the host. pos_in and
        seqlens_in are rows 0 and 1 of ps_in [2, B4] (B4 = B rounded up to 4,
        so that both rows start 16-byte aligned): one copy of a [2, B4] host
        tensor fills both. The graph keeps this cache's and these buffers'
        addresses and the kernels' launch parameters, so it is valid while
        they stay allocated. Run at least one eager step first (it sets the
        kernels' launch attributes)."""
        import torch
        dev = self.u.device
        b4 = (self.batch + 3) // 4 * 4
        self.h_in = torch.zeros((self.batch, self.shape.d), dtype=self.torch_dtype, device=dev)
        self.ps_in = torch.zeros((2, b4), dtype=torch.int32, device=dev)
        self.ps_in[1].fill_(1)
        self.pos_in = self.ps_in[0, :self.batch]
        self.seqlens_in = self.ps_in[1, :self.batch]
        torch.cuda.synchronize(dev)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            self.step(self.h_in, self.pos_in, cache, self.seqlens_in)
        self.graph = graph
        self.graph_launches = self.launches
        return graph

    def replay(self):
        """Run the captured step on the current stream; returns u [B, d]."""
        self.graph.replay()
        return self.u
