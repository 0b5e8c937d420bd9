"""Thin ctypes binding of libhybridattn.so (argument marshalling only).

Every function has the name of the C entry point it calls and takes torch
tensors (device memory) or raw integer device addresses.  The stream defaults to
torch's current CUDA stream.  A non-zero status raises HAError with the library's
own message.  If the shared library is missing, loading raises: there is no
fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libhybridattn.so")

F32, BF16 = 0, 1
ELIG_DISJOINT, ELIG_OVERLAP = 0, 1
OP_TOPK, OP_DECODE, OP_PREFILL, OP_DECODE_STEP = 0, 1, 2, 3
STATUS = {0: "HA_OK", 1: "HA_ERR_INVALID_ARG", 2: "HA_ERR_MISALIGNED", 3: "HA_ERR_UNSUPPORTED",
          4: "HA_ERR_WORKSPACE", 5: "HA_ERR_CUDA"}


class HAError(RuntimeError):
    def __init__(self, fn: str, code: int, detail: str):
        super().__init__(f"{fn}: {STATUS.get(code, code)}: {detail}")
        self.code = code


class Params(ctypes.Structure):
    """Mirror of ha_params (field order and types as in include/hybrid_attn.h)."""
    _fields_ = [("B", ctypes.c_int32), ("H", ctypes.c_int32), ("d", ctypes.c_int32),
                ("n_win", ctypes.c_int32), ("m", ctypes.c_int32), ("k", ctypes.c_int32),
                ("H_I", ctypes.c_int32), ("d_I", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("elig", ctypes.c_int32), ("scale", ctypes.c_float), ("fmt", ctypes.c_int32)]


FMT_KV8 = 1            # compressed K/V rows: RoPE dims bf16, the rest e4m3 (608 bytes)
FMT_IDX4 = 2           # FP4 indexer keys and queries, bfloat16 index scores
KV8_ROW_BYTES = 608    # one FP8 K or V row (d = 512)
IDX4_ROW_BYTES = 80    # one FP4 indexer key row (d_I = 128)


def make_params(B, H, d, n_win, m, k=1, H_I=1, d_I=8, dtype=BF16, elig=ELIG_DISJOINT, scale=0.0,
                fmt=0):
    return Params(B, H, d, n_win, m, k, H_I, d_I, dtype, elig, scale, fmt)


_P = ctypes.c_void_p
_I = ctypes.c_int32
_SZ = ctypes.c_size_t
_SIGS = {
    "hca_compress_kv": [ctypes.POINTER(Params), _P, _P, _P, _I, _P, _I, _P, _P, _I, _P],
    "csa_compress_kv": [ctypes.POINTER(Params), _P, _P, _P, _P, _I, _P, _I, _P, _P, _P, _I, _P],
    "csa_index_scores": [ctypes.POINTER(Params), _P, _P, _P, _I, _P, _I, _P, _P],
    "csa_topk": [ctypes.POINTER(Params), _P, _I, _P, _I, _P, _P, _SZ, _P],
    "hybrid_attn_decode": [ctypes.POINTER(Params), _P, _P, _P, _I, _P, _P, _P, _I, _P, _P, _P,
                           _P, _SZ, _P],
    "hybrid_attn_prefill": [ctypes.POINTER(Params), _P, _P, _I, _P, _P, _I, _P, _P, _P, _I, _P,
                            _P, _P, _SZ, _P],
    "csa_decode_step": [ctypes.POINTER(Params), _P, _P, _P, _P, _P, _P, _P, _I, _P, _P, _P, _P, _I,
                        _P, _P, _P, _P, _P, _SZ, _P],
    "hca_decode_step": [ctypes.POINTER(Params), _P, _P, _P, _P, _I, _P, _P, _P, _I, _P, _P, _P,
                        _SZ, _P],
    "hybrid_attn_decode_static": [ctypes.POINTER(Params), _P, _P, _P, _I, _P, _P, _P, _I, _P, _P,
                                  _P, _P],
    "hybrid_attn_merge": [ctypes.POINTER(Params), _I, _I, _P, _P, _P, _P, _P],
    "ha_workspace_size": [ctypes.POINTER(Params), _I, _I, _I, _I, ctypes.POINTER(ctypes.c_size_t)],
    "ha_device_error": [ctypes.POINTER(ctypes.c_int32), _I],
    "ha_selftest_wait_timeout": [_I, _P],
}
EXPORTS = list(_SIGS) + ["ha_status_string", "ha_last_error", "ha_abi_version", "ha_launch_count",
                         "ha_host_alloc", "ha_host_free"]

_lib = None


def load_library(path: str = LIB_PATH):
    """Load the CUDA library once; raises OSError when it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise OSError(f"{path} is missing: build it with python -m long_context_hybrid_02_b300.build")
    lib = ctypes.CDLL(path)
    for name, args in _SIGS.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    lib.ha_status_string.argtypes = [ctypes.c_int]
    lib.ha_status_string.restype = ctypes.c_char_p
    lib.ha_last_error.argtypes = []
    lib.ha_last_error.restype = ctypes.c_char_p
    lib.ha_abi_version.argtypes = []
    lib.ha_abi_version.restype = ctypes.c_int32
    lib.ha_launch_count.argtypes = []
    lib.ha_launch_count.restype = ctypes.c_uint64
    lib.ha_host_alloc.argtypes = [ctypes.c_size_t, ctypes.c_int32]
    lib.ha_host_alloc.restype = ctypes.c_void_p
    lib.ha_host_free.argtypes = [ctypes.c_void_p]
    lib.ha_host_free.restype = ctypes.c_int
    _lib = lib
    return lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _call(name, *args):
    lib = load_library()
    code = getattr(lib, name)(*args)
    if code != 0:
        raise HAError(name, code, lib.ha_last_error().decode())


def _ws(ws):
    if ws is None:
        return None, 0
    if isinstance(ws, tuple):
        return ws
    return ws.data_ptr(), ws.numel() * ws.element_size()


def hca_compress_kv(p, k_tok, v_tok, gate, tok_cap, blk_begin, n_blk, ck, cv, n_cap, stream=None):
    _call("hca_compress_kv", ctypes.byref(p), _ptr(k_tok), _ptr(v_tok), _ptr(gate), tok_cap,
          _ptr(blk_begin), n_blk, _ptr(ck), _ptr(cv), n_cap, _stream(stream))


def csa_compress_kv(p, k_tok, v_tok, ki_tok, gate, tok_cap, blk_begin, n_blk, ck, cv, cki, n_cap,
                    stream=None):
    _call("csa_compress_kv", ctypes.byref(p), _ptr(k_tok), _ptr(v_tok), _ptr(ki_tok), _ptr(gate),
          tok_cap, _ptr(blk_begin), n_blk, _ptr(ck), _ptr(cv), _ptr(cki), n_cap, _stream(stream))


def csa_index_scores(p, q_idx, w_idx, cki, n_cap, q_pos, Tq, scores, stream=None):
    _call("csa_index_scores", ctypes.byref(p), _ptr(q_idx), _ptr(w_idx), _ptr(cki), n_cap,
          _ptr(q_pos), Tq, _ptr(scores), _stream(stream))


def csa_topk(p, scores, n_cap, q_pos, Tq, idx, ws=None, stream=None):
    wp, wb = _ws(ws)
    _call("csa_topk", ctypes.byref(p), _ptr(scores), n_cap, _ptr(q_pos), Tq, _ptr(idx), wp, wb,
          _stream(stream))


def hybrid_attn_decode(p, q, ck, cv, n_cap, idx, k_tok, v_tok, tok_cap, ctx_len, o, lse=None,
                       ws=None, stream=None):
    wp, wb = _ws(ws)
    _call("hybrid_attn_decode", ctypes.byref(p), _ptr(q), _ptr(ck), _ptr(cv), n_cap, _ptr(idx),
          _ptr(k_tok), _ptr(v_tok), tok_cap, _ptr(ctx_len), _ptr(o), _ptr(lse), wp, wb,
          _stream(stream))


def hybrid_attn_merge(p, rows, S, o_part, lse_part, o, lse=None, stream=None):
    _call("hybrid_attn_merge", ctypes.byref(p), rows, S, _ptr(o_part), _ptr(lse_part), _ptr(o),
          _ptr(lse), _stream(stream))


def hybrid_attn_prefill(p, q, q_pos, Tq, ck, cv, n_cap, idx, k_tok, v_tok, tok_cap, o, lse=None,
                        ws=None, stream=None):
    wp, wb = _ws(ws)
    _call("hybrid_attn_prefill", ctypes.byref(p), _ptr(q), _ptr(q_pos), Tq, _ptr(ck), _ptr(cv),
          n_cap, _ptr(idx), _ptr(k_tok), _ptr(v_tok), tok_cap, _ptr(o), _ptr(lse), wp, wb,
          _stream(stream))


def csa_decode_step(p, q, q_idx, w_idx, k_tok, v_tok, ki_tok, gate, tok_cap, ctx_len, ck, cv,
                    cki, n_cap, scores, idx, o, lse=None, ws=None, stream=None):
    wp, wb = _ws(ws)
    _call("csa_decode_step", ctypes.byref(p), _ptr(q), _ptr(q_idx), _ptr(w_idx), _ptr(k_tok),
          _ptr(v_tok), _ptr(ki_tok), _ptr(gate), tok_cap, _ptr(ctx_len), _ptr(ck), _ptr(cv),
          _ptr(cki), n_cap, _ptr(scores), _ptr(idx), _ptr(o), _ptr(lse), wp, wb, _stream(stream))


def hca_decode_step(p, q, k_tok, v_tok, gate, tok_cap, ctx_len, ck, cv, n_cap, o, lse=None,
                    ws=None, stream=None):
    wp, wb = _ws(ws)
    _call("hca_decode_step", ctypes.byref(p), _ptr(q), _ptr(k_tok), _ptr(v_tok), _ptr(gate),
          tok_cap, _ptr(ctx_len), _ptr(ck), _ptr(cv), n_cap, _ptr(o), _ptr(lse), wp, wb,
          _stream(stream))


STATIC_SCRATCH_BYTES = 32 << 20


def hybrid_attn_decode_static(p, q, ck, cv, n_cap, idx, k_tok, v_tok, tok_cap, ctx_len, o,
                              lse=None, stream=None):
    """hybrid_attn_decode for callers that cannot allocate: no workspace argument,
    the library's fixed 32 MiB device scratch holds the split partials."""
    _call("hybrid_attn_decode_static", ctypes.byref(p), _ptr(q), _ptr(ck), _ptr(cv), n_cap,
          _ptr(idx), _ptr(k_tok), _ptr(v_tok), tok_cap, _ptr(ctx_len), _ptr(o), _ptr(lse),
          _stream(stream))


def ha_workspace_size(p, op, Tq, n_cap, is_csa) -> int:
    out = ctypes.c_size_t(0)
    _call("ha_workspace_size", ctypes.byref(p), op, Tq, n_cap, int(bool(is_csa)), ctypes.byref(out))
    return out.value


def ha_status_string(code: int) -> str:
    return load_library().ha_status_string(code).decode()


def ha_abi_version() -> int:
    return load_library().ha_abi_version()


def ha_launch_count() -> int:
    return load_library().ha_launch_count()


def host_empty(shape, dtype, write_combined: bool = False):
    """A CPU tensor of `shape` and `dtype` in page-locked memory from ha_host_alloc
    (released when the last tensor viewing it is gone).  Copies between it and the
    device run at the link's bandwidth; write_combined for inputs the host only
    writes."""
    import math
    import weakref

    import torch
    lib = load_library()
    nbytes = max(1, math.prod(shape)) * torch.empty((), dtype=dtype).element_size()
    ptr = lib.ha_host_alloc(nbytes, 1 if write_combined else 0)
    if not ptr:
        raise MemoryError(f"ha_host_alloc({nbytes}): {lib.ha_last_error().decode()}")
    buf = (ctypes.c_uint8 * nbytes).from_address(ptr)
    weakref.finalize(buf, lib.ha_host_free, ptr)
    return torch.frombuffer(buf, dtype=torch.uint8).view(dtype).reshape(shape)


def ha_device_error(clear: bool = True) -> int:
    """Error code recorded by a tensor-core kernel that gave up waiting (0 = none)."""
    code = ctypes.c_int32(0)
    _call("ha_device_error", ctypes.byref(code), int(clear))
    return code.value


def ha_selftest_wait_timeout(code: int, stream=None):
    """Launch the wait-timeout self-test: after the 2 s wait limit the device error
    word holds `code` (unless a code was already set)."""
    _call("ha_selftest_wait_timeout", code, _stream(stream))
