"""C-ABI library: it builds, loads, exports what include/specverify.h declares,
and rejects bad host-side arguments before launching anything.  No GPU."""

import ctypes
import os
import re

import pytest

from conftest import ROOT
from speculative_decoding_verification_temp_gb300 import _abi
from speculative_decoding_verification_temp_gb300 import build as build_mod

HEADER = os.path.join(ROOT, "include", "specverify.h")


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return _abi.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(spec_\w+)\s*\(", src)))


def test_header_declares_the_binding_exports():
    assert declared_functions() == sorted(_abi.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in (0, 1, 2, 3):
        assert _abi.status_string(code).startswith("SPEC_")
    assert "unknown" in _abi.status_string(42)


def test_workspace_size_rejects_bad_shapes(lib):
    assert lib.spec_verify_chain_workspace_size(4, 4, 0, 0) == 0
    assert lib.spec_verify_chain_workspace_size(4, 4, 100, 9) == 0
    assert lib.spec_verify_tree_workspace_size(4, 4, 100, 9) == 0


def test_workspace_sizes(lib):
    a = lib.spec_verify_chain_workspace_size(4, 4, 32000, 0)
    b = lib.spec_verify_chain_workspace_size(256, 7, 128256, 1)
    assert 0 < a < b
    assert lib.spec_verify_chain_workspace_size(-1, 4, 10, 0) == 0
    assert lib.spec_verify_tree_workspace_size(32, 60, 128256, 1) > 0
    assert lib.spec_verify_tree_workspace_size(1, -1, 10, 0) == 0


def test_tree_walk_workspace_holds_the_row_records(lib):
    # trees of at most 256 nodes take the rows stream and the walk: the
    # workspace holds one 64-bit record per consumer warp (8) per 32 KB chunk
    # of each of the 2N rows of a tree.  At V = 1,500,000 bf16 a 257-node tree
    # takes the resident kernel (beyond the streaming kernel's vocabulary),
    # whose workspace has no such records.
    T, V = 4, 1_500_000
    chunks = -(-V * 2 // 32768)  # bf16 rows of V entries in 32 KB chunks
    records = T * 2 * 256 * chunks * 8 * 8
    with_walk = lib.spec_verify_tree_workspace_size(T, 256, V, _abi.SPEC_BF16)
    without = lib.spec_verify_tree_workspace_size(T, 257, V, _abi.SPEC_BF16)
    assert with_walk >= records
    assert with_walk - without >= records * 0.9
    # at the tree workload's size the records fit the workspace as well
    assert lib.spec_verify_tree_workspace_size(32, 60, 128256, _abi.SPEC_BF16) >= \
        32 * 120 * 8 * 8 * 8


FAKE = ctypes.c_void_p(0x10000)  # never dereferenced: every call below fails its host checks


def policy():
    return _abi.spec_policy(FAKE.value, None)


def chain(lib, B=2, gamma=3, V=100, dtype=0, target=FAKE, ld_t=None, draft=FAKE, ld_d=None,
          tokens=FAKE, out=FAKE, ws=FAKE, ws_bytes=0, pol=None):
    pol = pol or policy()
    return lib.spec_verify_chain(target, ld_t if ld_t is not None else V, draft,
                                 ld_d if ld_d is not None else V, dtype, B, gamma, V, tokens,
                                 pol, pol, 1234, None, out, out, None, None, ws, ws_bytes, None)


def test_chain_rejects_bad_arguments(lib):
    INV = _abi.SPEC_ERR_INVALID_ARG
    assert chain(lib, B=-1) == INV
    assert chain(lib, gamma=-1) == INV
    assert chain(lib, gamma=4096) == INV
    assert chain(lib, V=0) == INV
    assert chain(lib, dtype=7) == INV
    assert chain(lib, target=None) == INV
    assert chain(lib, draft=None) == INV
    assert chain(lib, tokens=None) == INV
    assert chain(lib, out=None) == INV
    assert chain(lib, ws=None) == INV
    assert chain(lib, ld_t=99) == INV
    assert chain(lib, ld_d=50) == INV
    assert chain(lib, pol=_abi.spec_policy(None, None)) == INV
    # a workspace smaller than the query is rejected before any launch
    need = lib.spec_verify_chain_workspace_size(2, 3, 100, 0)
    assert chain(lib, ws_bytes=need - 1) == INV


def test_chain_empty_batch_is_a_no_op(lib):
    assert chain(lib, B=0, target=None, draft=None, tokens=None, out=None, ws=None) == _abi.SPEC_OK


def test_chain_unsupported_vocabulary(lib):
    # with top-k filtering a float32 row pair of 10^8 entries would have to fit
    # one cluster's shared memory: refused before any launch
    topk = _abi.spec_policy(FAKE.value, FAKE.value)
    assert chain(lib, V=100_000_000, pol=topk) == _abi.SPEC_ERR_UNSUPPORTED
    # without top-k the streaming chain path takes vocabularies up to
    # 2,097,152 entries (the draw kernel keeps 20 bytes per 256-entry step in
    # shared memory); this call's workspace (0 bytes) is too small for it
    assert lib.spec_verify_chain_workspace_size(2, 3, 2_097_152, 0) > 0
    assert chain(lib, V=2_097_152) == _abi.SPEC_ERR_INVALID_ARG
    # beyond that no kernel takes a float32 row: refused before any launch
    assert chain(lib, V=2_097_153) == _abi.SPEC_ERR_UNSUPPORTED
    assert chain(lib, V=100_000_000) == _abi.SPEC_ERR_UNSUPPORTED


def test_static_chain_refuses_before_any_cuda_call(lib):
    # B = 1024, gamma = 7 needs more workspace than the fixed scratch holds
    assert lib.spec_verify_chain_workspace_size(1024, 7, 128256, 1) > _abi.SPEC_STATIC_SCRATCH_BYTES
    assert lib.spec_verify_chain_workspace_size(256, 7, 128256, 1) < _abi.SPEC_STATIC_SCRATCH_BYTES
    pol = policy()
    args = (FAKE, 128256, FAKE, 128256, 1, 1024, 7, 128256, FAKE, pol, pol, 1, None,
            FAKE, FAKE, None, None, None)
    assert lib.spec_verify_chain_static(*args) == _abi.SPEC_ERR_UNSUPPORTED
    empty = (None, 0, None, 0, 1, 0, 7, 128256, None, pol, pol, 1, None, None, None, None, None,
             None)
    assert lib.spec_verify_chain_static(*empty) == _abi.SPEC_OK
    neg = (FAKE, 10, FAKE, 10, 1, -1, 7, 10, FAKE, pol, pol, 1, None, FAKE, FAKE, None, None, None)
    assert lib.spec_verify_chain_static(*neg) == _abi.SPEC_ERR_INVALID_ARG
    # the argument checks of spec_verify_chain come before the size limit
    INV = _abi.SPEC_ERR_INVALID_ARG
    for B, gamma, V, dtype in ((1024, 7, 0, 1), (1024, 4096, 128256, 1), (4, 7, 128256, 7),
                               (4, -1, 128256, 1)):
        a = (FAKE, max(V, 1), FAKE, max(V, 1), dtype, B, gamma, V, FAKE, pol, pol, 1, None,
             FAKE, FAKE, None, None, None)
        assert lib.spec_verify_chain_static(*a) == INV, (B, gamma, V, dtype)
    missing = (FAKE, 128256, FAKE, 128256, 1, 4, 7, 128256, None, pol, pol, 1, None,
               FAKE, FAKE, None, None, None)
    assert lib.spec_verify_chain_static(*missing) == INV  # no draft tokens


def test_static_scratch_size_matches_header():
    assert "#define SPEC_STATIC_SCRATCH_BYTES (16u * 1024u * 1024u)" in open(HEADER).read()
    assert _abi.SPEC_STATIC_SCRATCH_BYTES == 16 * 1024 * 1024


def tree(lib, T=2, N=5, V=100, max_depth=3, parent=FAKE, tokens=FAKE, out=FAKE, ws_bytes=0):
    pol = policy()
    return lib.spec_verify_tree(FAKE, V, FAKE, V, 1, T, N, V, max_depth, tokens, parent, pol, pol,
                                1, None, out, out, out, None, None, FAKE, ws_bytes, None)


def test_tree_rejects_bad_arguments(lib):
    INV = _abi.SPEC_ERR_INVALID_ARG
    assert tree(lib, N=0) == INV
    assert tree(lib, N=4097) == INV
    assert tree(lib, max_depth=-1) == INV
    assert tree(lib, T=-1) == INV
    assert tree(lib, parent=None) == INV
    assert tree(lib, tokens=None) == INV
    assert tree(lib, out=None) == INV
    assert tree(lib) == INV  # workspace too small
    assert tree(lib, T=0, parent=None, tokens=None, out=None) == _abi.SPEC_OK
    # aligned bf16 rows of 128 entries take the tree walk: a workspace one byte
    # short of the size query is refused before anything is launched
    need = lib.spec_verify_tree_workspace_size(2, 5, 128, _abi.SPEC_BF16)
    assert need > 0
    assert tree(lib, V=128, ws_bytes=need - 1) == INV


def test_mask_rejects_bad_arguments(lib):
    INV = _abi.SPEC_ERR_INVALID_ARG
    m = lib.spec_tree_mask
    assert m(FAKE, -1, 4, 2, FAKE, FAKE, None, None) == INV
    assert m(FAKE, 1, 0, 2, FAKE, FAKE, None, None) == INV
    assert m(FAKE, 1, 4097, 2, FAKE, FAKE, None, None) == INV
    assert m(FAKE, 1, 4, -1, FAKE, FAKE, None, None) == INV
    assert m(None, 1, 4, 2, FAKE, FAKE, None, None) == INV
    assert m(FAKE, 1, 4, 2, None, FAKE, None, None) == INV
    assert m(None, 0, 4, 2, None, None, None, None) == _abi.SPEC_OK


def test_flag_values_match_header():
    src = open(HEADER).read()
    for name in ("BAD_TOKEN", "ZERO_Q", "NONFINITE", "DEGENERATE_RESIDUAL", "DEPTH", "TIMEOUT",
                 "BAD_TREE"):
        m = re.search(rf"#define SPEC_FLAG_{name} (\d+)u", src)
        assert int(m.group(1)) == getattr(_abi, f"FLAG_{name}")


def test_library_links_no_torch(lib):
    """The library's dynamic dependencies (ELF NEEDED entries) name no torch library."""
    import shutil
    import subprocess
    if shutil.which("readelf") is None:
        pytest.skip("readelf not available")
    out = subprocess.run(["readelf", "-d", _abi.library_path()], capture_output=True,
                         text=True).stdout
    needed = re.findall(r"\(NEEDED\).*\[(.*)\]", out)
    assert needed and not any("torch" in n or "c10" in n for n in needed)


def overlap_call(lib, B=2, gamma=3, V=100, dtype=1, target=FAKE, draft=FAKE, out=FAKE, pol=None,
                 polq=None, ld=None):
    pol = pol or policy()
    polq = polq or pol
    return lib.spec_overlap(target, ld if ld is not None else V, draft,
                            ld if ld is not None else V, dtype, B, gamma, V, pol, polq, out, None,
                            None)


def test_overlap_rejects_bad_arguments(lib):
    INV = _abi.SPEC_ERR_INVALID_ARG
    assert overlap_call(lib, B=-1) == INV
    assert overlap_call(lib, gamma=-1) == INV
    assert overlap_call(lib, V=0) == INV
    assert overlap_call(lib, dtype=7) == INV
    assert overlap_call(lib, target=None) == INV
    assert overlap_call(lib, draft=None) == INV
    assert overlap_call(lib, out=None) == INV
    assert overlap_call(lib, ld=99) == INV
    assert overlap_call(lib, pol=_abi.spec_policy(None, None)) == INV
    # top-k policies are not supported by the overlap kernel
    topk = _abi.spec_policy(FAKE.value, FAKE.value)
    assert overlap_call(lib, polq=topk) == _abi.SPEC_ERR_UNSUPPORTED
    # nothing to compare: a no-op
    assert overlap_call(lib, B=0, target=None, draft=None, out=None) == _abi.SPEC_OK
    assert overlap_call(lib, gamma=0, target=None, draft=None, out=None) == _abi.SPEC_OK


def typical_call(lib, B=2, gamma=3, V=100, dtype=1, target=FAKE, tokens=FAKE, out=FAKE, pol=None,
                 ld=None, eps=0.1, delta=0.5, ws=FAKE, ws_bytes=None):
    pol = pol or policy()
    if ws_bytes is None:
        ws_bytes = lib.spec_typical_workspace_size(B, gamma, V, dtype)
    return lib.spec_typical_accept(target, ld if ld is not None else V, dtype, B, gamma, V, pol,
                                   tokens, eps, delta, out, out, None, ws, ws_bytes, None)


def test_typical_workspace_size(lib):
    # 256 bytes, 8 per row (rounded up to 256), 128 per 32 KB chunk of a row
    assert lib.spec_typical_workspace_size(3, 4, 100, 1) == 256 + 256 + 15 * 1 * 128
    assert lib.spec_typical_workspace_size(256, 7, 128256, 1) == 256 + 16384 + 2048 * 8 * 128
    assert lib.spec_typical_workspace_size(2, 1, 16385, 0) == 256 + 256 + 4 * 3 * 128
    assert lib.spec_typical_workspace_size(-1, 4, 100, 1) == 0
    assert lib.spec_typical_workspace_size(3, -1, 100, 1) == 0
    assert lib.spec_typical_workspace_size(3, 4, 0, 1) == 0
    assert lib.spec_typical_workspace_size(3, 4, 100, 9) == 0


def test_typical_rejects_bad_arguments(lib):
    INV = _abi.SPEC_ERR_INVALID_ARG
    assert typical_call(lib, B=-1) == INV
    assert typical_call(lib, gamma=-1) == INV
    assert typical_call(lib, V=0) == INV
    assert typical_call(lib, dtype=7) == INV
    assert typical_call(lib, target=None) == INV
    assert typical_call(lib, tokens=None) == INV
    assert typical_call(lib, out=None) == INV
    assert typical_call(lib, ld=99) == INV
    assert typical_call(lib, pol=_abi.spec_policy(None, None)) == INV
    assert typical_call(lib, eps=-0.1) == INV
    assert typical_call(lib, delta=float("nan")) == INV
    assert typical_call(lib, eps=float("inf")) == INV
    assert typical_call(lib, ws=None) == INV
    assert typical_call(lib, ws_bytes=8) == INV
    assert typical_call(lib, ws=ctypes.c_void_p(FAKE.value + 4)) == INV  # misaligned
    topk = _abi.spec_policy(FAKE.value, FAKE.value)
    assert typical_call(lib, pol=topk) == _abi.SPEC_ERR_UNSUPPORTED
    # nothing to verify: a no-op
    assert typical_call(lib, B=0, target=None, tokens=None, out=None, ws=None) == _abi.SPEC_OK


def test_tree_rerank_rejects_bad_arguments(lib):
    INV = _abi.SPEC_ERR_INVALID_ARG

    def call(T=2, N=10, m=3, par=FAKE, conf=FAKE, out=FAKE):
        return lib.spec_tree_rerank(par, conf, T, N, m, out, out, None, out, None, None)

    assert call(T=-1) == INV
    assert call(N=0) == INV
    assert call(N=4097) == INV
    assert call(m=0) == INV
    assert call(par=None) == INV
    assert call(conf=None) == INV
    assert call(out=None) == INV
    assert call(T=0, par=None, conf=None, out=None) == _abi.SPEC_OK


def test_binding_argtypes_match_the_header(lib):
    """Every function the header declares has as many parameters as the
    binding passes (a drift check for the ctypes argtypes)."""
    hdr = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    for name in _abi.EXPORTS:
        m = re.search(r"\b" + name + r"\s*\(([^)]*)\)\s*;", hdr)
        assert m, name
        params = [p for p in m.group(1).split(",") if p.strip() and p.strip() != "void"]
        argtypes = getattr(lib, name).argtypes
        assert argtypes is not None and len(argtypes) == len(params), (name, len(params))
