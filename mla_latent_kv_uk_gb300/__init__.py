"""Python binding of the GB300 absorbed-MLA decode library (libmla_gb300.so).

Argument marshalling only: every function below checks tensor devices,
dtypes and shapes, allocates outputs with torch when the caller passes none,
and calls the C entry point of the same name on torch's current CUDA stream.
All arithmetic runs in the library's CUDA kernels; there is no fallback.
Importing this module raises ImportError if the library has not been built
(``python -c "import __graft_entry__ as g; g.build()"``).
"""

from __future__ import annotations

import ctypes
import os

import torch

from . import _build

__all__ = [
    "MlaError", "BF16", "E4M3", "F32", "lib",
    "mla_version", "mla_status_string", "mla_get_device_error", "mla_selftest_wait_timeout",
    "mla_absorb_q", "mla_decode_workspace_size", "mla_decode_paged",
    "mla_decode_plan", "mla_merge_states", "mla_v_up", "mla_gather_cache",
    "mla_gather_cache_reorg", "mla_expand_kv", "mla_prefill_attn", "mla_rope_cache_write",
    "mla_stage_copy",
]

BF16, E4M3, F32 = 0, 1, 2
_DTYPE_CODE = {torch.bfloat16: BF16, torch.float8_e4m3fn: E4M3, torch.float32: F32}
_CODE_DTYPE = {v: k for k, v in _DTYPE_CODE.items()}

_p, _i, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t

_SIGNATURES = {
    "mla_status_string": ([_i], ctypes.c_char_p),
    "mla_version": ([], _i),
    "mla_get_device_error": ([ctypes.POINTER(_i), _p], _i),
    "mla_selftest_wait_timeout": ([ctypes.c_longlong, _p], _i),
    "mla_absorb_q": ([_p, _p, _p, _i, _i, _i, _f, _p, _p], _i),
    "mla_decode_workspace_size": ([_i, _i, _i, _i, _i, ctypes.POINTER(_sz)], _i),
    "mla_decode_paged": ([_p, _i, _f, _p, _i, _f, _p, _p, _p, _p, _i, _i, _i, _i,
                          _i, _f, _i, _i, _p, _i, _p, _p, _sz, _p], _i),
    "mla_decode_paged_noalloc": ([_p, _i, _f, _p, _i, _f, _p, _p, _p, _p, _i, _i, _i, _i,
                                  _i, _f, _i, _i, _p, _i, _p, _p], _i),
    "mla_decode_plan": ([_p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _i, _p, _sz, _p], _i),
    "mla_merge_states": ([_p, _i, _p, _i, _i, _i, _i, _p, _i, _p, _p], _i),
    "mla_v_up": ([_p, _p, _i, _i, _p, _p], _i),
    "mla_gather_cache": ([_p, _i, _f, _p, _p, _p, _p, _i, _i, _i, _i, _i, _p, _p], _i),
    "mla_gather_cache_reorg": ([_i, _i, _p, _p, _p, _i, _i, _f, _p, _i, _i, _i, _p,
                                _p, _p, _i, _p], _i),
    "mla_expand_kv": ([_p, _p, _i, _i, _p, _p, _p], _i),
    "mla_prefill_attn": ([_p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _f, _p, _p, _p], _i),
    "mla_rope_cache_write": ([_p, _p, _p, _p, _p, _i, _i, _f, _i, _p, _i, _f, _i, _p], _i),
    "mla_stage_copy": ([_p, _p, _sz, _p], _i),
}


def _load():
    path = _build.lib_path()
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build the CUDA library first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    handle = ctypes.CDLL(path)
    for name, (args, res) in _SIGNATURES.items():
        fn = getattr(handle, name)
        fn.argtypes = args
        fn.restype = res
    return handle


lib = _load()


class MlaError(RuntimeError):
    def __init__(self, fn, status):
        super().__init__(f"{fn}: {lib.mla_status_string(status).decode()} (status {status})")
        self.status = status


def _check(fn, status):
    if status != 0:
        raise MlaError(fn, status)


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _req(t, name, dtype=None, dims=None, device=True):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a tensor")
    if device and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise TypeError(f"{name}: dtype {t.dtype} not in {dtype}")
    if dims is not None and t.dim() != dims:
        raise ValueError(f"{name}: expected {dims} dims, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def mla_version() -> int:
    return lib.mla_version()


def mla_status_string(status: int) -> str:
    return lib.mla_status_string(status).decode()


def mla_get_device_error() -> int:
    code = _i(0)
    _check("mla_get_device_error", lib.mla_get_device_error(ctypes.byref(code), _stream()))
    return code.value


def mla_selftest_wait_timeout(limit_cycles):
    """Makes one bounded device wait run out (see include/mla.h)."""
    _check("mla_selftest_wait_timeout",
           lib.mla_selftest_wait_timeout(int(limit_cycles), _stream()))


def mla_absorb_q(q_nope, q_pe, w_uk_t, out_dtype=torch.bfloat16, q_scale=1.0, out=None):
    """q_nope [T,H,128], q_pe [T,H,64], w_uk_t [H,128,512] (bf16) -> q [T,H,576]."""
    _req(q_nope, "q_nope", torch.bfloat16, 3)
    T, H, _ = q_nope.shape
    _req(q_pe, "q_pe", torch.bfloat16, 3)
    _req(w_uk_t, "w_uk_t", torch.bfloat16, 3)
    if tuple(q_nope.shape) != (T, H, 128) or tuple(q_pe.shape) != (T, H, 64) \
            or tuple(w_uk_t.shape) != (H, 128, 512):
        raise ValueError("absorb shapes")
    if out is None:
        out = torch.empty((T, H, 576), dtype=out_dtype, device=q_nope.device)
    _req(out, "out", out_dtype, 3)
    _check("mla_absorb_q", lib.mla_absorb_q(_ptr(q_nope), _ptr(q_pe), _ptr(w_uk_t), T, H,
                                            _DTYPE_CODE[out_dtype], float(q_scale),
                                            _ptr(out), _stream()))
    return out


def mla_decode_workspace_size(B, q_len, H, max_seq_len, split_tiles=0) -> int:
    n = _sz(0)
    _check("mla_decode_workspace_size",
           lib.mla_decode_workspace_size(B, q_len, H, max_seq_len, split_tiles, ctypes.byref(n)))
    return n.value


def mla_decode_paged(q, kv_cache, block_table, seq_lens, *, sm_scale, q_scale=1.0,
                     k_scale=1.0, kv_starts=None, kv_ends=None, causal=True,
                     split_tiles=0, out_dtype=torch.bfloat16, out=None, lse=None,
                     workspace=None):
    """q [B,q_len,H,576], kv_cache [num_blocks,64,576] (bf16 or e4m3, same for both)
    -> (out [B,q_len,H,512], lse [B,q_len,H] fp32)."""
    _req(q, "q", (torch.bfloat16, torch.float8_e4m3fn), 4)
    B, q_len, H, D = q.shape
    _req(kv_cache, "kv_cache", q.dtype, 3)
    _req(block_table, "block_table", torch.int32, 2)
    _req(seq_lens, "seq_lens", torch.int32, 1)
    if D != 576 or tuple(kv_cache.shape[1:]) != (64, 576) or block_table.shape[0] != B \
            or seq_lens.shape[0] != B:
        raise ValueError("decode shapes")
    for name, t in (("kv_starts", kv_starts), ("kv_ends", kv_ends)):
        if t is not None:
            _req(t, name, torch.int32, 1)
    max_blocks = block_table.shape[1]
    if out is None:
        out = torch.empty((B, q_len, H, 512), dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, q_len, H), dtype=torch.float32, device=q.device)
    _req(out, "out", out_dtype, 4)
    _req(lse, "lse", torch.float32, 3)
    if workspace is None:
        n = mla_decode_workspace_size(B, q_len, H, max_blocks * 64, split_tiles)
        workspace = torch.empty(n, dtype=torch.uint8, device=q.device)
    _req(workspace, "workspace", torch.uint8, 1)
    _check("mla_decode_paged", lib.mla_decode_paged(
        _ptr(q), _DTYPE_CODE[q.dtype], float(q_scale), _ptr(kv_cache),
        _DTYPE_CODE[kv_cache.dtype], float(k_scale), _ptr(block_table), _ptr(seq_lens),
        _ptr(kv_starts), _ptr(kv_ends), B, q_len, H, max_blocks, kv_cache.shape[0],
        float(sm_scale), int(bool(causal)), int(split_tiles), _ptr(out),
        _DTYPE_CODE[out_dtype], _ptr(lse), _ptr(workspace), workspace.numel(), _stream()))
    return out, lse


def mla_decode_plan(seq_lens, B, q_len, H, max_blocks, *, kv_starts=None, kv_ends=None,
                    causal=True, kv_dtype=torch.bfloat16, split_tiles=0, n_groups=0):
    """Returns the int32 plan buffer (see include/mla.h)."""
    _req(seq_lens, "seq_lens", torch.int32, 1)
    J = B * q_len * ((H + 127) // 128)
    plan = torch.zeros(4 + 4 * (J + 1), dtype=torch.int32, device=seq_lens.device)
    _check("mla_decode_plan", lib.mla_decode_plan(
        _ptr(seq_lens), _ptr(kv_starts), _ptr(kv_ends), B, q_len, H, max_blocks,
        int(bool(causal)), _DTYPE_CODE[kv_dtype], split_tiles, n_groups, _ptr(plan),
        plan.numel() * 4, _stream()))
    return plan


def mla_merge_states(parts_out, parts_lse, out_dtype=None, out=None, out_lse=None):
    """parts_out [S,T,H,D], parts_lse [S,T,H] -> (out [T,H,D], lse [T,H])."""
    _req(parts_out, "parts_out", (torch.bfloat16, torch.float32), 4)
    S, T, H, D = parts_out.shape
    _req(parts_lse, "parts_lse", torch.float32, 3)
    if tuple(parts_lse.shape) != (S, T, H):
        raise ValueError("merge shapes")
    out_dtype = out_dtype or parts_out.dtype
    if out is None:
        out = torch.empty((T, H, D), dtype=out_dtype, device=parts_out.device)
    if out_lse is None:
        out_lse = torch.empty((T, H), dtype=torch.float32, device=parts_out.device)
    _req(out, "out", out_dtype, 3)
    _check("mla_merge_states", lib.mla_merge_states(
        _ptr(parts_out), _DTYPE_CODE[parts_out.dtype], _ptr(parts_lse), S, T, H, D,
        _ptr(out), _DTYPE_CODE[out_dtype], _ptr(out_lse), _stream()))
    return out, out_lse


def mla_v_up(o_lat, w_uv, out=None):
    """o_lat [T,H,512], w_uv [H,128,512] (bf16) -> [T,H,128] bf16."""
    _req(o_lat, "o_lat", torch.bfloat16, 3)
    T, H, _ = o_lat.shape
    _req(w_uv, "w_uv", torch.bfloat16, 3)
    if o_lat.shape[2] != 512 or tuple(w_uv.shape) != (H, 128, 512):
        raise ValueError("v_up shapes")
    if out is None:
        out = torch.empty((T, H, 128), dtype=torch.bfloat16, device=o_lat.device)
    _check("mla_v_up", lib.mla_v_up(_ptr(o_lat), _ptr(w_uv), T, H, _ptr(out), _stream()))
    return out


def mla_gather_cache(kv_cache, block_table, seq_lens, cu_out, total_rows, *,
                     seq_starts=None, k_scale=1.0, out_dtype=None, out=None):
    """Paged gather: out[cu_out[b]+j] = kv_cache[slot(b, seq_starts[b]+j)]."""
    _req(kv_cache, "kv_cache", (torch.bfloat16, torch.float8_e4m3fn), 3)
    _req(block_table, "block_table", torch.int32, 2)
    _req(seq_lens, "seq_lens", torch.int32, 1)
    _req(cu_out, "cu_out", torch.int32, 1)
    B = block_table.shape[0]
    out_dtype = out_dtype or kv_cache.dtype
    if out is None:
        out = torch.empty((total_rows, 576), dtype=out_dtype, device=kv_cache.device)
    _check("mla_gather_cache", lib.mla_gather_cache(
        _ptr(kv_cache), _DTYPE_CODE[kv_cache.dtype], float(k_scale), _ptr(block_table),
        _ptr(seq_lens), _ptr(seq_starts), _ptr(cu_out), B, block_table.shape[1],
        kv_cache.shape[0], int(total_rows), _DTYPE_CODE[out_dtype], _ptr(out), _stream()))
    return out


def mla_gather_cache_reorg(shard_caches, shard_block_tables, cu_out, total_rows, *,
                           interleave=1, k_scale=1.0, out_dtype=None, out=None,
                           padded_cu=None, rank_major_rows=0, rank_major_out=None):
    """Fused local gather + rank-major all-gather + reorg over W shards."""
    W = len(shard_caches)
    dt = shard_caches[0].dtype
    for k in range(W):
        _req(shard_caches[k], f"shard_caches[{k}]", dt, 3)
        _req(shard_block_tables[k], f"shard_block_tables[{k}]", torch.int32, 2)
    _req(cu_out, "cu_out", torch.int32, 1)
    B = shard_block_tables[0].shape[0]
    smb = shard_block_tables[0].shape[1]
    if any(t.shape != (B, smb) for t in shard_block_tables):
        raise ValueError("shard block tables must share one shape")
    out_dtype = out_dtype or dt
    dev = shard_caches[0].device
    if out is None:
        out = torch.empty((total_rows, 576), dtype=out_dtype, device=dev)
    if rank_major_rows and rank_major_out is None:
        rank_major_out = torch.empty((rank_major_rows, 576), dtype=out_dtype, device=dev)
    caches = (ctypes.c_void_p * W)(*[t.data_ptr() for t in shard_caches])
    tables = (ctypes.c_void_p * W)(*[t.data_ptr() for t in shard_block_tables])
    nbs = (ctypes.c_int * W)(*[t.shape[0] for t in shard_caches])
    _check("mla_gather_cache_reorg", lib.mla_gather_cache_reorg(
        W, interleave, ctypes.cast(caches, _p), ctypes.cast(tables, _p),
        ctypes.cast(nbs, _p), smb, _DTYPE_CODE[dt], float(k_scale), _ptr(cu_out), B,
        int(total_rows), _DTYPE_CODE[out_dtype], _ptr(out), _ptr(rank_major_out),
        _ptr(padded_cu), int(rank_major_rows), _stream()))
    return out, rank_major_out


def mla_expand_kv(kv_rows, w_kvb, H, k_out=None, v_out=None):
    """kv_rows [N,576], w_kvb [H*256,512] (bf16) -> (K [N,H,192], V [N,H,128])."""
    _req(kv_rows, "kv_rows", torch.bfloat16, 2)
    _req(w_kvb, "w_kvb", torch.bfloat16, 2)
    N = kv_rows.shape[0]
    if kv_rows.shape[1] != 576 or tuple(w_kvb.shape) != (H * 256, 512):
        raise ValueError("expand shapes")
    if k_out is None:
        k_out = torch.empty((N, H, 192), dtype=torch.bfloat16, device=kv_rows.device)
    if v_out is None:
        v_out = torch.empty((N, H, 128), dtype=torch.bfloat16, device=kv_rows.device)
    _check("mla_expand_kv", lib.mla_expand_kv(_ptr(kv_rows), _ptr(w_kvb), N, H,
                                              _ptr(k_out), _ptr(v_out), _stream()))
    return k_out, v_out


def mla_prefill_attn(q, k, v, cu_q, cu_k, max_q_len, *, causal, sm_scale, out=None, lse=None):
    """q [Tq,H,192], k [Nk,H,192], v [Nk,H,128] -> (out [Tq,H,128] bf16, lse [Tq,H])."""
    _req(q, "q", torch.bfloat16, 3)
    _req(k, "k", torch.bfloat16, 3)
    _req(v, "v", torch.bfloat16, 3)
    _req(cu_q, "cu_q", torch.int32, 1)
    _req(cu_k, "cu_k", torch.int32, 1)
    Tq, H, _ = q.shape
    Nk = k.shape[0]
    B = cu_q.shape[0] - 1
    if q.shape[2] != 192 or tuple(k.shape) != (Nk, H, 192) or tuple(v.shape) != (Nk, H, 128):
        raise ValueError("prefill shapes")
    if out is None:
        out = torch.empty((Tq, H, 128), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((Tq, H), dtype=torch.float32, device=q.device)
    _check("mla_prefill_attn", lib.mla_prefill_attn(
        _ptr(q), _ptr(k), _ptr(v), _ptr(cu_q), _ptr(cu_k), B, Tq, Nk, H, int(max_q_len),
        int(bool(causal)), float(sm_scale), _ptr(out), _ptr(lse), _stream()))
    return out, lse


_ROPE_LAYOUT = {"interleaved": 0, "half": 1}


def mla_rope_cache_write(q_pe, k_pe, kv_c, positions, slot_mapping, kv_cache, *,
                         rope_base=10000.0, layout="interleaved", k_scale=1.0):
    """Rotates q_pe [T,H,64] (or None) and k_pe [T,64] (bf16) in place by
    positions [T] and stores kv_c [T,512] ‖ k_pe into kv_cache
    [num_blocks,64,576] (bf16 or e4m3) at slot_mapping [T] (int32)."""
    _req(k_pe, "k_pe", torch.bfloat16, 2)
    _req(kv_c, "kv_c", torch.bfloat16, 2)
    _req(positions, "positions", torch.int32, 1)
    _req(slot_mapping, "slot_mapping", torch.int32, 1)
    _req(kv_cache, "kv_cache", (torch.bfloat16, torch.float8_e4m3fn), 3)
    T = k_pe.shape[0]
    H = 0
    if q_pe is not None:
        _req(q_pe, "q_pe", torch.bfloat16, 3)
        if q_pe.shape[0] != T or q_pe.shape[2] != 64:
            raise ValueError("q_pe must be [T, H, 64]")
        H = q_pe.shape[1]
    if (k_pe.shape[1] != 64 or tuple(kv_c.shape) != (T, 512) or positions.shape[0] != T
            or slot_mapping.shape[0] != T or tuple(kv_cache.shape[1:]) != (64, 576)):
        raise ValueError("rope / cache-write shapes")
    _check("mla_rope_cache_write", lib.mla_rope_cache_write(
        _ptr(q_pe), _ptr(k_pe), _ptr(kv_c), _ptr(positions), _ptr(slot_mapping), T, H,
        float(rope_base), _ROPE_LAYOUT[layout], _ptr(kv_cache), _DTYPE_CODE[kv_cache.dtype],
        float(k_scale), kv_cache.shape[0], _stream()))


def mla_stage_copy(dst, src):
    """Copies src into dst (same byte size, both contiguous): exactly one of
    them a CUDA tensor of the current device, the other a pinned CPU tensor.
    The library's SMs move the bytes over the host link.  Returns dst."""
    for t, name in ((dst, "dst"), (src, "src")):
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if dst.is_cuda == src.is_cuda:
        raise ValueError("exactly one of dst, src must be a CUDA tensor")
    host = src if dst.is_cuda else dst
    if not host.is_pinned():
        raise ValueError("the host tensor must be pinned (page-locked)")
    nbytes = dst.numel() * dst.element_size()
    if nbytes != src.numel() * src.element_size():
        raise ValueError("dst and src differ in size")
    _check("mla_stage_copy", lib.mla_stage_copy(_ptr(dst), _ptr(src), nbytes, _stream()))
    return dst
