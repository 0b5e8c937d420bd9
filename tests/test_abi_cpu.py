"""The C-ABI library loads, exports every entry point of include/hybrid_attn.h and
rejects bad arguments on the host (no GPU needed: validation runs before any
CUDA call)."""
import os
import re

import pytest

from long_context_hybrid_02_b300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "hybrid_attn.h")


def header_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*([a-z_0-9]+)\s*\(",
                                 src, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    from long_context_hybrid_02_b300 import build as bld
    bld.build()
    return B.load_library()


def test_every_header_symbol_is_exported(lib):
    names = header_functions()
    assert {"hca_compress_kv", "csa_compress_kv", "csa_index_scores", "csa_topk",
            "hybrid_attn_decode", "hybrid_attn_prefill"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(B.EXPORTS)


def test_host_alloc_refuses_zero_bytes_and_frees_null(lib):
    assert lib.ha_host_alloc(0, 0) is None
    assert b"bytes = 0" in lib.ha_last_error()
    assert lib.ha_host_free(None) == 0


def test_version_and_status_strings(lib):
    assert B.ha_abi_version() == 3
    for code in range(6):
        assert B.ha_status_string(code) not in ("", "unknown status")
    assert B.ha_status_string(99) == "unknown status"


def P(**kw):
    base = dict(B=2, H=8, d=64, n_win=128, m=4, k=16, H_I=2, d_I=32, dtype=B.F32)
    base.update(kw)
    return B.make_params(**base)


A = 1 << 20      # a 16-byte aligned fake address (never dereferenced: the calls fail first)


def code_of(fn, *args):
    with pytest.raises(B.HAError) as e:
        fn(*args)
    return e.value.code


def test_compress_validation(lib):
    blk = A
    assert code_of(B.hca_compress_kv, P(), None, A, A, 1024, blk, 1, A, A, 256, 0) == 1
    assert code_of(B.hca_compress_kv, P(), A + 4, A, A, 1024, blk, 1, A, A, 256, 0) == 2
    assert code_of(B.hca_compress_kv, P(d=60), A, A, A, 1024, blk, 1, A, A, 256, 0) == 3
    assert code_of(B.hca_compress_kv, P(m=2000), A, A, A, 4096, blk, 1, A, A, 256, 0) == 3
    assert code_of(B.hca_compress_kv, P(), A, A, A, 2, blk, 1, A, A, 256, 0) == 1
    assert code_of(B.csa_compress_kv, P(d_I=12), A, A, A, A, 1024, blk, 1, A, A, A, 256, 0) == 3
    assert code_of(B.csa_compress_kv, P(), A, A, None, A, 1024, blk, 1, A, A, A, 256, 0) == 1
    assert code_of(B.csa_compress_kv, P(), A, A, A, A, 1024, blk, -1, A, A, A, 256, 0) == 1
    # n_blk == 0 is a no-op that returns before any CUDA call
    B.hca_compress_kv(P(), A, A, A, 1024, blk, 0, A, A, 256, 0)


def test_index_topk_validation(lib):
    assert code_of(B.csa_index_scores, P(H_I=0), A, A, A, 256, A, 1, A, 0) == 3
    assert code_of(B.csa_index_scores, P(H_I=128, d_I=512), A, A, A, 256, A, 1, A, 0) == 3
    assert code_of(B.csa_index_scores, P(), A, A, A, 0, A, 1, A, 0) == 1
    assert code_of(B.csa_index_scores, P(), A, A, A, 256, A, 0, A, 0) == 1
    assert code_of(B.csa_index_scores, P(), A + 8, A, A, 256, A, 1, A, 0) == 2
    assert code_of(B.csa_index_scores, P(), A, A + 2, A, 256, A, 1, A, 0) == 2
    assert code_of(B.csa_topk, P(k=0), A, 256, A, 1, A, None, 0) == 3
    assert code_of(B.csa_topk, P(k=5000), A, 256, A, 1, A, None, 0) == 3
    assert code_of(B.csa_topk, P(dtype=7), A, 256, A, 1, A, None, 0) == 1
    assert code_of(B.csa_topk, P(elig=3), A, 256, A, 1, A, None, 0) == 1
    assert code_of(B.csa_topk, P(), A, 40960 * 1024 + 1, A, 1, A, None, 0) == 3
    ws_long = B.ha_workspace_size(P(), B.OP_TOPK, 1, 262144, True)
    # 2 rows cut into 148 segments in all (one CTA per SM on a B300), each with a
    # (count, threshold) pair and a list of at most 2,048 (key, index) candidates
    assert ws_long == 148 * (8 + 2048 * 8)
    assert code_of(B.csa_topk, P(), A, 262144, A, 1, A, (A, ws_long - 1), 0) == 4


def test_attention_validation(lib):
    ws_need = B.ha_workspace_size(P(), B.OP_DECODE, 1, 256, True)
    assert ws_need > 0
    assert code_of(B.hybrid_attn_decode, P(), A, A, A, 256, A, A, A, 1024, A, A, None,
                   (A, ws_need - 1), 0) == 4
    assert code_of(B.hybrid_attn_decode, P(), A, A, A, 256, A, A, A, 1024, A, A, None,
                   None, 0) == 4
    assert code_of(B.hybrid_attn_decode, P(H=300), A, A, A, 256, A, A, A, 1024, A, A, None,
                   (A, ws_need), 0) == 3
    assert code_of(B.hybrid_attn_decode, P(), A, A, A, 256, A, A, A, 64, A, A, None,
                   (A, ws_need), 0) == 1          # tok_cap < n_win
    assert code_of(B.hybrid_attn_decode, P(), A, A, A, 256, A, A, A, 1024, None, A, None,
                   (A, ws_need), 0) == 1          # ctx_len NULL
    assert code_of(B.hybrid_attn_decode, P(scale=float("nan")), A, A, A, 256, A, A, A, 1024,
                   A, A, None, (A, ws_need), 0) == 1
    assert code_of(B.hybrid_attn_prefill, P(), A, A, 0, A, A, 256, A, A, A, 1024, A, None,
                   None, 0) == 1
    assert code_of(B.hybrid_attn_prefill, P(), A, A, 4, A, A, 256, A + 2, A, A, 1024, A, None,
                   None, 0) == 2


def test_attention_workspace_holds_the_split_partials(lib):
    """The tensor-core decode attention cuts every row's key list into S splits
    when the rows are too few to fill the GPU (S = floor(148 / (rows x H/64)), at
    least 32 keys per split, keys per split rounded up to 16); each split's float32
    o and lse per head go through the workspace: rows x S x H x (512 + 1) floats.
    On a machine without a GPU the plan assumes 148 SMs, as on the B300."""
    def ws(Bn, H, n_cap, csa, k=1024):
        p = B.make_params(Bn, H, 512, 128, 4 if csa else 128, k if csa else 1,
                          64 if csa else 1, 128 if csa else 8, B.BF16)
        return B.ha_workspace_size(p, B.OP_DECODE, 1, n_cap, csa)
    # 64K CSA (k = 512): 32 rows x 4 splits of 160 keys (512 + 128)
    assert ws(32, 64, 16384, True, k=512) == 32 * 4 * 64 * 513 * 4
    assert ws(160, 64, 1024, False) == 0         # 160 rows >= 148 SMs: one split each
    # 128K HCA: 32 rows x 4 splits of 288 keys (1,024 + 128 -> 1,152)
    assert ws(32, 64, 1024, False) == 32 * 4 * 64 * 513 * 4
    # 1M CSA: 4 rows x 2 head groups; 18 splits of 64 keys (1,024 + 128)
    assert ws(4, 128, 262144, True) == 4 * 18 * 128 * 513 * 4
    # 1M HCA: 18 splits of 464 keys (8,192 + 128)
    assert ws(4, 128, 8192, False) == 4 * 18 * 128 * 513 * 4


def test_workspace_sizes(lib):
    # decode partials grow with the key list; HCA lists are n_cap + n_win long
    a = B.ha_workspace_size(P(), B.OP_DECODE, 1, 256, True)
    b = B.ha_workspace_size(P(), B.OP_DECODE, 1, 4096, False)
    assert b >= a > 0
    assert B.ha_workspace_size(P(), B.OP_TOPK, 1, 256, True) == 0      # one CTA per row
    assert B.ha_workspace_size(P(), B.OP_TOPK, 1, 40960, True) == 0
    assert B.ha_workspace_size(P(), B.OP_TOPK, 1, 40961, True) > 0
    with pytest.raises(B.HAError):
        B.ha_workspace_size(P(), 9, 1, 256, True)
    with pytest.raises(B.HAError):
        B.ha_workspace_size(P(), B.OP_DECODE, 0, 256, True)


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(OSError):
        B.load_library.__wrapped__(str(tmp_path / "nope.so")) if hasattr(B.load_library, "__wrapped__") \
            else _load_fresh(str(tmp_path / "nope.so"))


def _load_fresh(path):
    saved = B._lib
    B._lib = None
    try:
        return B.load_library(path)
    finally:
        B._lib = saved


def test_wait_timeout_selftest_checks_its_code_on_the_host(lib):
    # rejected before any CUDA call: runs without a GPU
    assert code_of(B.ha_selftest_wait_timeout, 0, 0) == 1
    assert code_of(B.ha_selftest_wait_timeout, -5, 0) == 1
    assert "positive" in B.load_library().ha_last_error().decode()
