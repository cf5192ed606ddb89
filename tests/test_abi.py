"""C ABI checks that need no GPU: the library builds for sm_103a, loads, exports
every symbol the header declares, and rejects bad arguments before any launch."""

import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sba.h")

needs_nvcc = pytest.mark.skipif(shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"),
                                reason="nvcc not available")


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"SBA_API\s+[\w\s\*]+?\b(sba_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from selected_block_attention_gb300 import _build
    import selected_block_attention_gb300 as sba

    _build.build()
    return sba.load_library()


def test_header_declares_expected_entry_points():
    import selected_block_attention_gb300 as sba

    assert _declared() == sorted(sba.EXPORTED_SYMBOLS)


@needs_nvcc
def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name
    assert lib.sba_version().decode().startswith("sba ")


@needs_nvcc
def test_argument_validation_without_launch(lib):
    c = ctypes
    fake = c.c_void_p(0x10000)  # never dereferenced: validation fails first
    # null pointers
    r = lib.sba_nsa_select_fwd(None, None, None, None, None, None, 16, 16, None, 0, 1, 64, 4, 1, 128,
                               64, 1, 0.0, 0, None, None, None)
    assert r == -1 and b"null" in lib.sba_last_error()
    # unsupported head dim
    r = lib.sba_nsa_select_fwd(fake, fake, fake, None, fake, None, 16, 16, None, 0, 1, 64, 4, 1, 96,
                               64, 1, 0.0, 0, fake, None, None)
    assert r == -2 and b"D must be" in lib.sba_last_error()
    # Hq not a multiple of Hkv
    r = lib.sba_nsa_select_fwd(fake, fake, fake, None, fake, None, 16, 16, None, 0, 1, 64, 6, 4, 128,
                               64, 1, 0.0, 0, fake, None, None)
    assert r == -1
    # misaligned pointer
    r = lib.sba_nsa_select_fwd(c.c_void_p(0x10002), fake, fake, None, fake, None, 16, 16, None, 0, 1, 64,
                               4, 1, 128, 64, 1, 0.0, 0, fake, None, None)
    assert r == -1 and b"aligned" in lib.sba_last_error()
    # varlen with B > 1
    r = lib.sba_nsa_select_fwd(fake, fake, fake, None, fake, None, 16, 16, fake, 3, 2, 64, 4, 1, 128,
                               64, 1, 0.0, 0, fake, None, None)
    assert r == -1
    # bounds: window below -1
    r = lib.sba_sparse_mask_bounds(fake, fake, fake, fake, 1, 64, 64, 16, 16, 1, -2, 0, -1, fake,
                                   fake, fake, fake, None)
    assert r == -1
    r = lib.sba_sparse_mask_dkdv_bounds(fake, fake, fake, fake, 1, 64, 64, 16, 16, 1, -2, 0, -1,
                                        fake, fake, fake, fake, None)
    assert r == -1
    r = lib.sba_sparse_mask_dkdv_bounds(fake, fake, fake, fake, 1, 64, 64, 16, 8192, 1, -1, -1,
                                        -1, fake, fake, fake, fake, None)
    assert r == -2
    r = lib.sba_sparse_mask_dkdv_bounds(fake, None, fake, fake, 1, 64, 64, 16, 16, 1, -1, -1, -1,
                                        fake, fake, fake, fake, None)
    assert r == -1 and b"null" in lib.sba_last_error()
    # block-sparse: q_block must be 128
    r = lib.sba_blocksparse_attn_fwd(fake, fake, fake, fake, fake, fake, fake, fake, fake, fake,
                                     fake, 1, 256, 4, 2, 128, 64, 64, 1, -1, -1, -1, 0.0, fake,
                                     None, None)
    assert r == -2
    # decode: workspace too small
    need = lib.sba_ragged_decode_workspace_size(4, 8, 1024, 128, -1)
    assert need > 0
    r = lib.sba_ragged_decode_fwd(fake, fake, fake, fake, fake, 4, 8, 2, 1024, 128, 0.0, -1, -1,
                                  0.0, None, 0, 0, fake, None, fake, need - 1, None)
    assert r == -1 and b"workspace" in lib.sba_last_error()
    # decode: too many sinks
    r = lib.sba_ragged_decode_fwd(fake, fake, fake, fake, fake, 4, 8, 2, 1024, 128, 0.0, -1, -1,
                                  0.0, fake, 17, 1, fake, None, fake, need, None)
    assert r == -2
    assert lib.sba_ragged_decode_workspace_size(0, 8, 1024, 128, -1) == 0
    # multi-query: workspace too small, unsupported head dim, Q < 1, too many sinks
    need = lib.sba_ragged_flash_attention_workspace_size(4, 3, 8, 1024, 128, 100, 0)
    assert need > 0
    args = [fake, fake, fake, fake, fake, 4, 3, 8, 2, 1024, 128, 0.0, 100, 0, 0.0, None, 0, 0,
            fake, None, fake, need - 1, None]
    assert lib.sba_ragged_flash_attention_fwd(*args) == -1
    assert b"workspace" in lib.sba_last_error()
    args[-2] = need
    args[10] = 64
    assert lib.sba_ragged_flash_attention_fwd(*args) == -2
    args[10] = 128
    args[6] = 0
    assert lib.sba_ragged_flash_attention_fwd(*args) == -1
    args[6] = 3
    args[15], args[16] = fake, 17
    assert lib.sba_ragged_flash_attention_fwd(*args) == -2
    assert lib.sba_ragged_flash_attention_workspace_size(4, 0, 8, 1024, 128, 100, 0) == 0
    # host-buffer NSA entry: null host pointer, misaligned / short workspace, unsupported D
    need = lib.sba_nsa_select_host_workspace_size(2, 64, 4, 2, 128, 4, 0, 1, 0, 1)
    assert need > 0
    hargs = [fake, fake, fake, None, fake, fake, 0, 4, 2, 64, 4, 2, 128, 64, 1, 0.0, 0, fake, fake,
             c.c_void_p(0x100000), need, None]
    r = lib.sba_nsa_select_fwd_host(None, *hargs[1:])
    assert r == -1 and b"null" in lib.sba_last_error()
    hargs[19] = c.c_void_p(0x100010)
    assert lib.sba_nsa_select_fwd_host(*hargs) == -1 and b"aligned" in lib.sba_last_error()
    hargs[19] = c.c_void_p(0x100000)
    hargs[20] = need - 1
    assert lib.sba_nsa_select_fwd_host(*hargs) == -1 and b"workspace" in lib.sba_last_error()
    hargs[20] = need
    hargs[12] = 96
    assert lib.sba_nsa_select_fwd_host(*hargs) == -2
    assert lib.sba_nsa_select_host_workspace_size(0, 64, 4, 2, 128, 4, 0, 1, 0, 1) == 0
    # L2 probe: misaligned buffer, size not a multiple of 16, no sink
    assert lib.sba_l2_read_probe(c.c_void_p(0x10008), 4096, 1, fake, None) == -1
    assert lib.sba_l2_read_probe(fake, 4100, 1, fake, None) == -1
    assert lib.sba_l2_read_probe(fake, 4096, 1, None, None) == -1
    assert lib.sba_l2_read_probe(fake, 4096, 0, fake, None) == -1


def test_workspace_size_grows_with_window():
    """Host-only arithmetic of the workspace query (library built or not)."""
    import selected_block_attention_gb300 as sba

    try:
        lib = sba.load_library()
    except RuntimeError:
        pytest.skip("library not built")
    a = lib.sba_ragged_decode_workspace_size(64, 32, 32768, 128, 4096)
    b = lib.sba_ragged_decode_workspace_size(64, 32, 32768, 128, -1)
    assert 0 < a < b


def test_multi_query_workspace_arithmetic():
    """Split count of the multi-query workspace (1024 keys per split) and its split
    counters: a 16-row tile
    spans queries i_lo..i_hi (at most 16), so its key range is at most
    left + min(Q, right + 16) keys with both window bounds, left + Q with only a left
    bound, S without one; Q = 1 gives the decode workspace."""
    import selected_block_attention_gb300 as sba

    try:
        lib = sba.load_library()
    except RuntimeError:
        pytest.skip("library not built")
    ws = lib.sba_ragged_flash_attention_workspace_size

    def expect(B, Q, Hq, splits):
        # fp32 partials (D + 2 per row, split, query, head) rounded up to 256 bytes, then
        # one int counter per (batch row, KV head, 16-row tile): at most
        # ceil(Q * Hq / 16) + Hq per batch row whatever Hkv is
        partials = B * splits * Q * Hq * (128 + 2) * 4
        return (partials + 255) // 256 * 256 + B * ((Q * Hq + 15) // 16 + Hq) * 4

    assert ws(64, 4, 32, 32768, 128, 4096, 0) == expect(64, 4, 32, 5)     # 4100 keys
    assert ws(64, 4, 32, 32768, 128, 4096, -1) == expect(64, 4, 32, 5)
    assert ws(64, 4, 32, 32768, 128, -1, 0) == expect(64, 4, 32, 32)
    assert ws(64, 4, 32, 32768, 128, 1020, 0) == expect(64, 4, 32, 1)     # 1024 keys
    assert ws(64, 4, 32, 32768, 128, 1021, 0) == expect(64, 4, 32, 2)     # 1025 keys
    assert ws(2, 64, 32, 32768, 128, 1000, 8) == expect(2, 64, 32, 1)     # 1000 + 24 keys
    assert ws(2, 64, 32, 32768, 128, 1000, -1) == expect(2, 64, 32, 2)    # 1000 + 64 keys
    assert ws(2, 64, 32, 32768, 128, 1000, 40) == expect(2, 64, 32, 2)    # 1000 + 56 keys
    assert ws(2, 64, 32, 32768, 128, 1000, 60) == expect(2, 64, 32, 2)    # 1000 + 64 keys
    assert ws(2, 64, 32, 1000, 128, -1, 60) == expect(2, 64, 32, 1)       # S = 1000
    for wl in (-1, 0, 4096, 5000):
        assert ws(64, 1, 32, 32768, 128, wl, 7) == lib.sba_ragged_decode_workspace_size(64, 32, 32768, 128, wl)


def test_nsa_host_workspace_arithmetic():
    """Staging layout of the host-buffer NSA entry: q, k, v, indices, counts, gate, out,
    lse for all rows, each rounded up to 256 bytes (host-only arithmetic)."""
    import selected_block_attention_gb300 as sba

    try:
        lib = sba.load_library()
    except RuntimeError:
        pytest.skip("library not built")
    r = lambda x: (x + 255) // 256 * 256
    B, T, Hq, Hkv, D, S = 3, 100, 4, 2, 64, 5
    q = B * T * Hq * D * 2
    kv = B * T * Hkv * D * 2
    full = r(q) + 2 * r(kv) + r(B * T * Hkv * S * 4) + r(B * T * Hkv * 4) + r(B * T * Hq * 2) + r(q) + r(B * T * Hq * 4)
    assert lib.sba_nsa_select_host_workspace_size(B, T, Hq, Hkv, D, S, 0, 1, 1, 1) == full
    bare = r(q) + 2 * r(kv) + r(B * T * Hkv * S * 4) + r(q)
    assert lib.sba_nsa_select_host_workspace_size(B, T, Hq, Hkv, D, S, 0, 0, 0, 0) == bare
    f32 = 2 * r(2 * q) + 2 * r(2 * kv) + r(B * T * Hkv * S * 4) + r(B * T * Hq * 4)
    assert lib.sba_nsa_select_host_workspace_size(B, T, Hq, Hkv, D, S, 1, 0, 0, 1) == f32
    assert lib.sba_nsa_select_host_workspace_size(B, T, Hq, Hkv, D, S, 7, 0, 0, 1) == 0
