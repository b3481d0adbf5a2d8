"""mla_decode_paged_noalloc, the decode entry point that allocates nothing,
against mla_decode_paged with a caller workspace.

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

pytestmark = pytest.mark.gpu

OUT_TOL, LSE_TOL = 1e-2, 1e-3   # the decode tolerances of the other tests


def _i32(x):
    return torch.as_tensor(np.asarray(x, dtype=np.int32)).cuda()


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    import mla_latent_kv_uk_gb300 as m
    case = synth.decode_case("noalloc", 700, B=5, H=128,
                             seq_lens=[1, 33, 700, 2500, 4096], q_len=1, poison=True)
    q, cache = case.q.cuda(), case.cache.cuda()
    bt, sl = _i32(case.block_table), _i32(case.seq_lens)
    ref_o, ref_l = m.mla_decode_paged(q, cache, bt, sl, sm_scale=case.sm_scale)
    torch.cuda.synchronize()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):
        out = torch.full_like(ref_o, float("nan"))
        lse = torch.full_like(ref_l, float("nan"))
        st = m.lib.mla_decode_paged_noalloc(
            _p(q), m.BF16, 1.0, _p(cache), m.BF16, 1.0, _p(bt), _p(sl), None, None,
            case.B, case.q_len, case.H, case.block_table.shape[1], cache.shape[0],
            case.sm_scale, 1, 0, _p(out), m.BF16, _p(lse), stream)
        assert st == 0, m.mla_status_string(st)
        torch.cuda.synchronize()
        d_o = (out.float() - ref_o.float()).abs().max().item()
        d_l = (lse - ref_l).abs().max().item()
        assert d_o <= OUT_TOL and d_l <= LSE_TOL, (d_o, d_l)
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
