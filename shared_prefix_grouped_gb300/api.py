"""Python binding of the grouped-attention C ABI.  Torch supplies device memory and streams only;
every step of the computation runs in the library's CUDA kernels.

    layout = pack(prefix_lens, group_sizes, suffix_lens)          # pg_pack
    o, lse = grouped_attn_fwd(layout, q, k, v, rope_theta=1e4)     # pg_grouped_attn_fwd
    dq, dk, dv = grouped_attn_bwd(layout, q, k, v, o, lse, do)    # pg_grouped_attn_bwd
"""
from __future__ import annotations

import ctypes as C
from typing import Optional, Sequence

import torch

from . import _lib
from ._lib import PgLayout, PgOpts, check, int_array

_DT = {torch.float32: _lib.PG_F32, torch.bfloat16: _lib.PG_BF16}


def _stream_ptr(device: torch.device) -> C.c_void_p:
    return C.c_void_p(torch.cuda.current_stream(device).cuda_stream)


class Layout:
    """A packed batch: the C layout struct plus the device buffers it points into."""

    def __init__(self, prefix_lens, group_sizes, suffix_lens, struct: PgLayout,
                 position_ids: torch.Tensor, tables: torch.Tensor):
        self.prefix_lens = list(prefix_lens)
        self.group_sizes = list(group_sizes)
        self.suffix_lens = list(suffix_lens)
        self.struct = struct
        self.position_ids = position_ids
        self.tables = tables

    @property
    def total_tokens(self) -> int:
        return int(self.struct.total_tokens)

    @property
    def pairs(self) -> int:
        return int(self.struct.pairs)


def pack_size(prefix_lens, group_sizes, suffix_lens):
    T, nb = C.c_int64(), C.c_int64()
    check("pg_pack_size", _lib.lib().pg_pack_size(
        len(prefix_lens), int_array(prefix_lens), int_array(group_sizes), int_array(suffix_lens),
        C.byref(T), C.byref(nb)))
    return T.value, nb.value


def pack_host(prefix_lens: Sequence[int], group_sizes: Sequence[int], suffix_lens: Sequence[int]):
    """Host-only packing (no CUDA): returns (position_ids int32 tensor, tables uint8 tensor, struct)."""
    T, nb = pack_size(prefix_lens, group_sizes, suffix_lens)
    pos = torch.empty(T, dtype=torch.int32)
    tab = torch.empty(nb, dtype=torch.uint8)
    st = PgLayout()
    check("pg_pack_host", _lib.lib().pg_pack_host(
        len(prefix_lens), int_array(prefix_lens), int_array(group_sizes), int_array(suffix_lens),
        C.cast(pos.data_ptr(), _lib.I32P), C.c_void_p(tab.data_ptr()), nb, C.byref(st)))
    return pos, tab, st


def pack(prefix_lens: Sequence[int], group_sizes: Sequence[int], suffix_lens: Sequence[int],
         device="cuda") -> Layout:
    device = torch.device(device)
    T, nb = pack_size(prefix_lens, group_sizes, suffix_lens)
    pos = torch.empty(T, dtype=torch.int32, device=device)
    tab = torch.empty(nb, dtype=torch.uint8, device=device)
    st = PgLayout()
    with torch.cuda.device(device):
        check("pg_pack", _lib.lib().pg_pack(
            len(prefix_lens), int_array(prefix_lens), int_array(group_sizes),
            int_array(suffix_lens), C.c_void_p(pos.data_ptr()), C.c_void_p(tab.data_ptr()), nb,
            C.byref(st), _stream_ptr(device)))
    return Layout(prefix_lens, group_sizes, suffix_lens, st, pos, tab)


def pack_tree_size(parent: Sequence[int], seg_lens: Sequence[int]):
    T, nb = C.c_int64(), C.c_int64()
    check("pg_pack_tree_size", _lib.lib().pg_pack_tree_size(
        len(parent), int_array(parent), int_array(seg_lens), C.byref(T), C.byref(nb)))
    return T.value, nb.value


def pack_tree_host(parent: Sequence[int], seg_lens: Sequence[int]):
    """Host-only packing of nested prefixes: (position_ids, tables, struct), as pack_host."""
    T, nb = pack_tree_size(parent, seg_lens)
    pos = torch.empty(T, dtype=torch.int32)
    tab = torch.empty(nb, dtype=torch.uint8)
    st = PgLayout()
    check("pg_pack_tree_host", _lib.lib().pg_pack_tree_host(
        len(parent), int_array(parent), int_array(seg_lens), C.cast(pos.data_ptr(), _lib.I32P),
        C.c_void_p(tab.data_ptr()), nb, C.byref(st)))
    return pos, tab, st


def pack_tree(parent: Sequence[int], seg_lens: Sequence[int], device="cuda") -> Layout:
    """Layout of nested prefixes: segments in depth-first preorder, parent[i] = -1 for a root."""
    device = torch.device(device)
    T, nb = pack_tree_size(parent, seg_lens)
    pos = torch.empty(T, dtype=torch.int32, device=device)
    tab = torch.empty(nb, dtype=torch.uint8, device=device)
    st = PgLayout()
    with torch.cuda.device(device):
        check("pg_pack_tree", _lib.lib().pg_pack_tree(
            len(parent), int_array(parent), int_array(seg_lens), C.c_void_p(pos.data_ptr()),
            C.c_void_p(tab.data_ptr()), nb, C.byref(st), _stream_ptr(device)))
    lay = Layout([], [], [], st, pos, tab)
    lay.tree = (list(parent), list(seg_lens))
    return lay


def _padded_args(num_groups, prefix_len, group_size, max_response_len, response_lens):
    assert len(response_lens) == num_groups * group_size
    return (int(num_groups), int(prefix_len), int(group_size), int(max_response_len),
            int_array(response_lens))


def pack_padded_size(num_groups: int, prefix_len: int, group_size: int, max_response_len: int,
                     response_lens: Sequence[int]):
    T, nb = C.c_int64(), C.c_int64()
    check("pg_pack_padded_size", _lib.lib().pg_pack_padded_size(
        *_padded_args(num_groups, prefix_len, group_size, max_response_len, response_lens),
        C.byref(T), C.byref(nb)))
    return T.value, nb.value


def pack_padded_host(num_groups: int, prefix_len: int, group_size: int, max_response_len: int,
                     response_lens: Sequence[int]):
    """Host-only padded packing: (position_ids, tables, struct), as pack_host."""
    T, nb = pack_padded_size(num_groups, prefix_len, group_size, max_response_len, response_lens)
    pos = torch.empty(T, dtype=torch.int32)
    tab = torch.empty(nb, dtype=torch.uint8)
    st = PgLayout()
    check("pg_pack_padded_host", _lib.lib().pg_pack_padded_host(
        *_padded_args(num_groups, prefix_len, group_size, max_response_len, response_lens),
        C.cast(pos.data_ptr(), _lib.I32P), C.c_void_p(tab.data_ptr()), nb, C.byref(st)))
    return pos, tab, st


def pack_padded(num_groups: int, prefix_len: int, group_size: int, max_response_len: int,
                response_lens: Sequence[int], device="cuda") -> Layout:
    """Layout of a padded batch [P; slot_1; ...; slot_G] per group (slots of max_response_len
    tokens, response i in the first response_lens[i] of its slot); attention calls on it write
    zeros (and lse = +inf) on the padding rows."""
    device = torch.device(device)
    T, nb = pack_padded_size(num_groups, prefix_len, group_size, max_response_len, response_lens)
    pos = torch.empty(T, dtype=torch.int32, device=device)
    tab = torch.empty(nb, dtype=torch.uint8, device=device)
    st = PgLayout()
    with torch.cuda.device(device):
        check("pg_pack_padded", _lib.lib().pg_pack_padded(
            *_padded_args(num_groups, prefix_len, group_size, max_response_len, response_lens),
            C.c_void_p(pos.data_ptr()), C.c_void_p(tab.data_ptr()), nb, C.byref(st),
            _stream_ptr(device)))
    return Layout([prefix_len] * num_groups, [group_size] * num_groups,
                  [max_response_len] * (num_groups * group_size), st, pos, tab)


def make_opts(rope_theta: float = 0.0, softmax_scale: float = 0.0, flags: int = 0,
              debug: int = 0) -> PgOpts:
    return PgOpts(float(softmax_scale), float(rope_theta), int(flags), int(debug))


def _dims(q: torch.Tensor, k: torch.Tensor):
    if q.dim() != 3 or k.dim() != 3:
        raise ValueError("q must be [T, Hq, d] and k, v [T, Hkv, d]")
    return q.shape[1], k.shape[1], q.shape[2]


def _ptr(t: Optional[torch.Tensor]) -> C.c_void_p:
    return C.c_void_p(t.data_ptr() if t is not None else 0)


def _contig(*ts):
    for t in ts:
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("tensors must be contiguous CUDA tensors")


def workspace_size(layout: Layout, dtype: torch.dtype, Hq: int, Hkv: int, d: int, opts: PgOpts,
                   phase: int) -> int:
    n = C.c_size_t()
    check("pg_workspace_size", _lib.lib().pg_workspace_size(
        C.byref(layout.struct), _DT[dtype], Hq, Hkv, d, C.byref(opts), phase, C.byref(n)))
    return n.value


def _workspace(n: int, device) -> torch.Tensor:
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device)


def grouped_attn_fwd(layout: Layout, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, *,
                     rope_theta: float = 0.0, softmax_scale: float = 0.0, flags: int = 0,
                     debug: int = 0, out: Optional[torch.Tensor] = None,
                     lse: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None):
    Hq, Hkv, d = _dims(q, k)
    _contig(q, k, v)
    opts = make_opts(rope_theta, softmax_scale, flags, debug)
    T = layout.total_tokens
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((Hq, T), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = _workspace(workspace_size(layout, q.dtype, Hq, Hkv, d, opts, 0), q.device)
    with torch.cuda.device(q.device):
        check("pg_grouped_attn_fwd", _lib.lib().pg_grouped_attn_fwd(
            C.byref(layout.struct), _DT[q.dtype], Hq, Hkv, d, _ptr(q), _ptr(k), _ptr(v),
            _ptr(out), _ptr(lse), C.byref(opts), _ptr(workspace), workspace.numel(),
            _stream_ptr(q.device)))
    return out, lse


def grouped_attn_bwd(layout: Layout, q, k, v, o, lse, do, *, rope_theta: float = 0.0,
                     softmax_scale: float = 0.0, flags: int = 0, debug: int = 0,
                     dq: Optional[torch.Tensor] = None, dk: Optional[torch.Tensor] = None,
                     dv: Optional[torch.Tensor] = None,
                     workspace: Optional[torch.Tensor] = None):
    Hq, Hkv, d = _dims(q, k)
    _contig(q, k, v, o, lse, do)
    opts = make_opts(rope_theta, softmax_scale, flags, debug)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if workspace is None:
        workspace = _workspace(workspace_size(layout, q.dtype, Hq, Hkv, d, opts, 1), q.device)
    with torch.cuda.device(q.device):
        check("pg_grouped_attn_bwd", _lib.lib().pg_grouped_attn_bwd(
            C.byref(layout.struct), _DT[q.dtype], Hq, Hkv, d, _ptr(q), _ptr(k), _ptr(v), _ptr(o),
            _ptr(lse), _ptr(do), _ptr(dq), _ptr(dk), _ptr(dv), C.byref(opts), _ptr(workspace),
            workspace.numel(), _stream_ptr(q.device)))
    return dq, dk, dv


def rope_table(layout: Layout, dtype: torch.dtype, Hq: int, Hkv: int, d: int,
               workspace: torch.Tensor, *, rope_theta: float, flags: int) -> int:
    """Writes the cos/sin table of PG_FLAG_PRE_ROTATED into `workspace` (pg_rope_table) and
    returns its device address; flags must include PG_FLAG_PRE_ROTATED."""
    opts = make_opts(rope_theta, 0.0, flags)
    table = C.c_void_p()
    with torch.cuda.device(workspace.device):
        check("pg_rope_table", _lib.lib().pg_rope_table(
            C.byref(layout.struct), _DT[dtype], Hq, Hkv, d, C.byref(opts), _ptr(workspace),
            workspace.numel(), C.byref(table), _stream_ptr(workspace.device)))
    return int(table.value)


def gemm_bf16_rope(a: torch.Tensor, b: torch.Tensor, table: int, table_rows: int, head_dim: int,
                   out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """bf16 [M, N] = a [M, K] @ b [N, K]^T with every head_dim-wide column block RoPE-rotated in
    the epilogue by the rows' (cos, sin) from `table` (pg_gemm_bf16_rope)."""
    if a.dtype != torch.bfloat16 or b.dtype != torch.bfloat16:
        raise ValueError("gemm_bf16_rope takes bf16 operands")
    _contig(a, b)
    M, K = a.shape
    N, Kb = b.shape
    if K != Kb:
        raise ValueError("inner dimensions differ")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=a.device)
    if out.dtype != torch.bfloat16 or out.dim() != 2 or out.stride(1) != 1 or out.shape != (M, N):
        raise ValueError("out must be a bf16 [M, N] matrix with unit column stride")
    with torch.cuda.device(a.device):
        check("pg_gemm_bf16_rope", _lib.lib().pg_gemm_bf16_rope(
            M, N, K, _ptr(a), a.shape[1], _ptr(b), b.shape[1], _ptr(out), out.stride(0), head_dim,
            C.c_void_p(table), table_rows, _stream_ptr(a.device)))
    return out


def device_status(clear: bool = True) -> int:
    """The kernels' status word (0 = ok); synchronous."""
    return int(_lib.lib().pg_device_status(1 if clear else 0))


def gemm_bf16(a: torch.Tensor, b: torch.Tensor, *, a_mn: bool = False, b_mn: bool = False,
              out_dtype: torch.dtype = torch.float32, out: Optional[torch.Tensor] = None,
              accumulate: bool = False):
    """C[m, n] = sum_k A(m, k) B(n, k) on the tensor cores (pg_gemm_bf16).

    a is [M, K] (a_mn False) or [K, M] (a_mn True); b is [N, K] (b_mn False) or [K, N] (True).
    """
    if a.dtype != torch.bfloat16 or b.dtype != torch.bfloat16:
        raise ValueError("gemm_bf16 takes bf16 operands")
    _contig(a, b)
    M, K = (a.shape[1], a.shape[0]) if a_mn else (a.shape[0], a.shape[1])
    N, Kb = (b.shape[1], b.shape[0]) if b_mn else (b.shape[0], b.shape[1])
    if K != Kb:
        raise ValueError("inner dimensions differ")
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=a.device)
    if out.dim() != 2 or out.stride(1) != 1 or not out.is_cuda or out.shape != (M, N):
        raise ValueError("out must be a [M, N] CUDA matrix with unit column stride")
    with torch.cuda.device(a.device):
        check("pg_gemm_bf16", _lib.lib().pg_gemm_bf16(
            M, N, K, _ptr(a), int(a_mn), a.shape[1], _ptr(b), int(b_mn), b.shape[1], _ptr(out),
            _DT[out.dtype], out.stride(0), int(accumulate), _stream_ptr(a.device)))
    return out


def rmsnorm_fwd(x: torch.Tensor, gamma: torch.Tensor, eps: float, residual=None):
    """out = rmsnorm(x [+ residual]) * gamma; returns (out, y, rstd) with y the normalised input."""
    _contig(x, gamma)
    T, H = x.shape
    out = torch.empty_like(x)
    y = torch.empty_like(x) if residual is not None else x
    rstd = torch.empty(T, dtype=torch.float32, device=x.device)
    with torch.cuda.device(x.device):
        check("pg_rmsnorm_fwd", _lib.lib().pg_rmsnorm_fwd(
            T, H, _ptr(x), _ptr(residual), _ptr(gamma), float(eps), _ptr(out),
            _ptr(y if residual is not None else None), _ptr(rstd), _stream_ptr(x.device)))
    return out, y, rstd


def rmsnorm_bwd(y, gamma, rstd, dout, dres=None, dx_dtype=torch.bfloat16):
    """Returns (dx, dgamma)."""
    T, H = y.shape
    dx = torch.empty((T, H), dtype=dx_dtype, device=y.device)
    dgamma = torch.empty(H, dtype=torch.float32, device=y.device)
    L = _lib.lib()
    nws = L.pg_rmsnorm_bwd_workspace(T, H)
    ws = _workspace(nws, y.device)
    with torch.cuda.device(y.device):
        check("pg_rmsnorm_bwd", L.pg_rmsnorm_bwd(
            T, H, _ptr(y), _ptr(gamma), _ptr(rstd), _ptr(dout), _DT[dout.dtype], _ptr(dres),
            _ptr(dx), _DT[dx_dtype], _ptr(dgamma), _ptr(ws), ws.numel(), _stream_ptr(y.device)))
    return dx, dgamma


def swiglu_fwd(gate_up: torch.Tensor):
    T, I2 = gate_up.shape
    out = torch.empty((T, I2 // 2), dtype=gate_up.dtype, device=gate_up.device)
    with torch.cuda.device(gate_up.device):
        check("pg_swiglu_fwd", _lib.lib().pg_swiglu_fwd(T, I2 // 2, _ptr(gate_up), _ptr(out),
                                                         _stream_ptr(gate_up.device)))
    return out


def swiglu_bwd(gate_up: torch.Tensor, dout: torch.Tensor):
    T, I2 = gate_up.shape
    dgu = torch.empty_like(gate_up)
    with torch.cuda.device(gate_up.device):
        check("pg_swiglu_bwd", _lib.lib().pg_swiglu_bwd(T, I2 // 2, _ptr(gate_up), _ptr(dout),
                                                         _ptr(dgu), _stream_ptr(gate_up.device)))
    return dgu
