"""CPU checks of the C ABI: the library builds/loads, exports every function
include/mla.h declares, and rejects bad arguments on the host before any
launch (no GPU needed for any of these calls)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _lib_path():
    import __graft_entry__ as entry
    b = entry._build_module()
    if not os.path.exists(b.lib_path()):
        b.build()
    return b.lib_path()


def _declared():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"\b(mla_\w+)\s*\(", src)
    return sorted(set(names))


def test_header_declares_the_path():
    names = _declared()
    for want in ["mla_absorb_q", "mla_decode_paged", "mla_decode_plan",
                 "mla_decode_workspace_size", "mla_merge_states", "mla_v_up",
                 "mla_gather_cache", "mla_gather_cache_reorg", "mla_expand_kv",
                 "mla_prefill_attn", "mla_rope_cache_write", "mla_status_string",
                 "mla_get_device_error"]:
        assert want in names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(_lib_path())
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings_and_version():
    _lib_path()
    import mla_latent_kv_uk_gb300 as m
    assert m.mla_version() == 1
    assert m.mla_status_string(0) == "ok"
    assert "workspace" in m.mla_status_string(3)
    assert m.mla_status_string(999) == "unknown status"


def test_host_validation_rejects_bad_arguments():
    import mla_latent_kv_uk_gb300 as m
    L = m.lib
    s = ctypes.c_void_p(0)
    # bounded-wait self-test: the limit must be 1 .. 1e9 cycles
    assert L.mla_selftest_wait_timeout(0, s) == 1
    assert L.mla_selftest_wait_timeout(2 * 10 ** 9, s) == 1
    # merge: S = 0, D not a multiple of 8, bad dtype
    assert L.mla_merge_states(None, 0, None, 0, 1, 1, 8, None, 0, None, s) == 1
    assert L.mla_merge_states(None, 0, None, 2, 1, 1, 12, None, 0, None, s) == 1
    assert L.mla_merge_states(None, 7, None, 2, 1, 1, 8, None, 0, None, s) == 1
    # absorb: negative T, bad out dtype, fp8 with zero scale
    assert L.mla_absorb_q(None, None, None, -1, 1, 0, 1.0, None, s) == 1
    assert L.mla_absorb_q(None, None, None, 1, 1, 9, 1.0, None, s) == 1
    assert L.mla_absorb_q(None, None, None, 1, 1, 1, 0.0, None, s) == 1
    # absorb with T == 0 is a no-op even with null pointers
    assert L.mla_absorb_q(None, None, None, 0, 1, 0, 1.0, None, s) == 0
    # decode: B = 0, mixed q/kv dtypes, null pointers
    args = [None, 0, 1.0, None, 0, 1.0, None, None, None, None, 0, 1, 128, 1, 1,
            0.1, 1, 0, None, 0, None, None, 0, s]
    assert L.mla_decode_paged(*args) == 1
    args[10] = 1
    assert L.mla_decode_paged(*args) == 1          # null q
    # gather: e4m3 -> f32 is not a supported conversion
    assert L.mla_gather_cache(None, 1, 1.0, None, None, None, None, 1, 1, 1, 1, 2,
                              None, s) == 1
    # reorg: W out of range
    assert L.mla_gather_cache_reorg(17, 1, None, None, None, 1, 0, 1.0, None, 1, 0,
                                    0, None, None, None, 0, s) == 1
    # rope / cache write: bad layout, base <= 1, e4m3 with zero scale, null
    # pointers; T == 0 is a no-op
    assert L.mla_rope_cache_write(None, None, None, None, None, 1, 0, 10000.0, 2,
                                  None, 0, 1.0, 1, s) == 1
    assert L.mla_rope_cache_write(None, None, None, None, None, 1, 0, 1.0, 0,
                                  None, 0, 1.0, 1, s) == 1
    assert L.mla_rope_cache_write(None, None, None, None, None, 1, 0, 10000.0, 0,
                                  None, 1, 0.0, 1, s) == 1
    assert L.mla_rope_cache_write(None, None, None, None, None, 1, 0, 10000.0, 0,
                                  None, 0, 1.0, 1, s) == 1
    assert L.mla_rope_cache_write(None, None, None, None, None, 0, 0, 10000.0, 0,
                                  None, 0, 1.0, 1, s) == 0
    # host staging: null pointers, a size that is not a multiple of 16, an
    # unaligned pointer; zero bytes is a no-op
    assert L.mla_stage_copy(None, None, 16, s) == 1
    assert L.mla_stage_copy(ctypes.c_void_p(4096), ctypes.c_void_p(8192), 24, s) == 1
    assert L.mla_stage_copy(ctypes.c_void_p(4100), ctypes.c_void_p(8192), 16, s) == 1
    assert L.mla_stage_copy(None, None, 0, s) == 0


def test_workspace_size_grows_with_work():
    import mla_latent_kv_uk_gb300 as m
    a = m.mla_decode_workspace_size(1, 1, 128, 4096)
    b = m.mla_decode_workspace_size(32, 1, 128, 4096)
    c = m.mla_decode_workspace_size(32, 1, 128, 4096, split_tiles=4)
    assert 0 < a < b < c
    with pytest.raises(m.MlaError):
        m.mla_decode_workspace_size(0, 1, 128, 4096)


@pytest.mark.parametrize("B,q_len,H,max_seq,split", [(3, 1, 128, 1000, 1), (5, 2, 200, 4096, 7),
                                                     (32, 1, 128, 4096, 3), (9, 4, 16, 64, 2)])
def test_workspace_covers_every_split_the_plan_format_allows(B, q_len, H, max_seq, split):
    """mla_decode_workspace_size (host only) must hold the plan and one fp32
    partial (128 x 512) plus its 128 LSEs for every segment a forced split
    can produce, worst case: every request at the maximum length.  From the
    plan format documented with mla_decode_plan: a job of n key tiles of 64
    takes n + 4 units, spans are C = split units long, and the spans meet at
    most J + spans - 1 (job, span) pairs (each span boundary cuts one job)."""
    import mla_latent_kv_uk_gb300 as m
    HG = (H + 127) // 128
    J = B * q_len * HG
    units = J * ((max_seq + 63) // 64 + 4)
    spans = -(-units // split)
    segs = J + spans - 1
    plan_bytes = (4 + 4 * (J + 1)) * 4
    need = plan_bytes + segs * (128 * 512 * 4 + 128 * 4)
    got = m.mla_decode_workspace_size(B, q_len, H, max_seq, split)
    assert got >= need
    # and not grossly more (the bound is within one slot per job of this)
    assert got <= need + (J + 2) * (128 * 512 * 4 + 128 * 4) + 4096
