"""mla_decode_paged_noalloc, the decode entry point that allocates nothing,
against mla_decode_paged with a caller workspace and against the oracle.

Callers that cannot allocate device memory at call time (serving runtimes
whose device memory is carved up once before traffic starts, plug-in hosts
that forbid allocation on the call path, plain C hosts without an allocator)
use the no-allocation entry point: its scratch is a static device array
inside the library.  This file is named so pytest
collects it after every other test file."""

import ctypes

import numpy as np
import pytest
import torch

import synth
from oracle import mla as O
from tests._helpers import check_attention, decode_terms, f64

pytestmark = pytest.mark.gpu

OUT_TOL, LSE_TOL = 1e-2, 1e-3   # the decode tolerances of the other tests


def _i32(x):
    return torch.as_tensor(np.asarray(x, dtype=np.int32)).cuda()


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc(m, q, cache, bt, sl, case, out, lse, stream, B=None, q_len=None, H=None):
    return m.lib.mla_decode_paged_noalloc(
        _p(q), m.BF16, 1.0, _p(cache), m.BF16, 1.0, _p(bt), _p(sl), None, None,
        case.B if B is None else B, case.q_len if q_len is None else q_len,
        case.H if H is None else H, case.block_table.shape[1], cache.shape[0],
        case.sm_scale, 1, 0, _p(out), m.BF16, _p(lse), stream)


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    import mla_latent_kv_uk_gb300 as m
    case = synth.decode_case("noalloc", 700, B=5, H=128,
                             seq_lens=[1, 33, 700, 2500, 4096], q_len=1, poison=True)
    q, cache = case.q.cuda(), case.cache.cuda()
    bt, sl = _i32(case.block_table), _i32(case.seq_lens)
    ref_o, ref_l = m.mla_decode_paged(q, cache, bt, sl, sm_scale=case.sm_scale)
    torch.cuda.synchronize()
    q64, c64 = f64(case.q), f64(case.cache)
    oo, ol = O.paged_decode(q64, c64, case.block_table, case.seq_lens, case.sm_scale)
    t = decode_terms(q64, c64, case.block_table, case.seq_lens, case.sm_scale)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    out = torch.full_like(ref_o, float("nan"))
    lse = torch.full_like(ref_l, float("nan"))
    for call in range(2):
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        st = _noalloc(m, q, cache, bt, sl, case, out, lse, stream)
        assert st == 0, m.mla_status_string(st)
        torch.cuda.synchronize()
        if call == 1:
            # the promise of this entry point: a call takes no device memory
            assert torch.cuda.mem_get_info()[0] == free_before
        d_o = (out.float() - ref_o.float()).abs().max().item()
        d_l = (lse - ref_l).abs().max().item()
        assert d_o <= OUT_TOL and d_l <= LSE_TOL, (d_o, d_l)
        check_attention(f64(out), lse.cpu().numpy(), oo, ol, t, out_tol=OUT_TOL,
                        lse_tol=LSE_TOL, label=f"noalloc call {call}")
    assert m.mla_get_device_error() == 0


def test_noalloc_rejects_requests_beyond_its_scratch():
    import mla_latent_kv_uk_gb300 as m
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    dummy = torch.zeros(16, dtype=torch.uint8, device="cuda")
    p = _p(dummy)
    # 4096 requests x 2048 pages need far more than the 64 MiB scratch
    st = m.lib.mla_decode_paged_noalloc(p, m.BF16, 1.0, p, m.BF16, 1.0, p, p, None, None,
                                        4096, 1, 128, 2048, 1, 0.07, 1, 0, p, m.BF16, p,
                                        stream)
    assert st == 3 and "workspace" in m.mla_status_string(st)
    # the argument checks come first: a null query is a bad argument
    st = m.lib.mla_decode_paged_noalloc(None, m.BF16, 1.0, p, m.BF16, 1.0, p, p, None, None,
                                        4096, 1, 128, 2048, 1, 0.07, 1, 0, p, m.BF16, p,
                                        stream)
    assert st == 1
    # the spec-decode shape (B = 128, q_len 2, H = 128: 256 jobs) does not fit
    st = m.lib.mla_decode_paged_noalloc(p, m.BF16, 1.0, p, m.BF16, 1.0, p, p, None, None,
                                        128, 2, 128, 512, 1, 0.07, 1, 0, p, m.BF16, p,
                                        stream)
    assert st == 3
    # the DeepSeek-V3 decode shape does (checked on the host only: the
    # workspace query of the same shape is within the scratch)
    assert m.mla_decode_workspace_size(32, 1, 128, 4096) <= 64 * 1024 * 1024
