"""The allocation-free forward entry point (pg_grouped_attn_fwd_noalloc), called through the C ABI,
against the regular entry point (pg_grouped_attn_fwd) on the same inputs.

It serves callers that may not allocate device memory themselves; its scratch is a fixed array the
library reserves on each GPU.  This file is collected last so that a run stopping at the first
failure has run every other test first; it also passes when run alone in a fresh process.
"""
import ctypes as C

import pytest
import torch

from oracle import prefix_grouper_oracle as orc
from shared_prefix_grouped_gb300 import _lib, api, workloads
from shared_prefix_grouped_gb300.build import build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build()


def call_noalloc(layout, q, k, v, o, lse, theta):
    opts = api.make_opts(theta)
    Hq, Hkv, d = q.shape[1], k.shape[1], q.shape[2]
    return _lib.lib().pg_grouped_attn_fwd_noalloc(
        C.byref(layout.struct), _lib.PG_BF16, Hq, Hkv, d, C.c_void_p(q.data_ptr()),
        C.c_void_p(k.data_ptr()), C.c_void_p(v.data_ptr()), C.c_void_p(o.data_ptr()),
        C.c_void_p(lse.data_ptr()), C.byref(opts),
        C.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_forward_matches_regular_entry_point_twice():
    base = workloads.WORKLOADS[2]
    dev = torch.device("cuda")
    for seed in (11, 12):       # two calls in a row share (and overwrite) the same scratch
        w = workloads.small_variant(base, prefix_len=300, suffix_lens=[64, 1, 200, 129],
                                    heads_q=8, heads_kv=2, seed=seed)
        prob = workloads.make_problem(w)
        lay = api.pack(prob.prefix_lens, prob.group_sizes, prob.suffix_lens, dev)
        q, k, v = (t.to(dev) for t in (prob.q, prob.k, prob.v))
        o_ref, lse_ref = api.grouped_attn_fwd(lay, q, k, v, rope_theta=w.rope_theta)
        o = torch.full_like(q, float("nan"))
        lse = torch.full_like(lse_ref, float("nan"))
        assert call_noalloc(lay, q, k, v, o, lse, w.rope_theta) == _lib.PG_OK
        torch.cuda.synchronize()
        assert api.device_status() == 0
        assert orc.normwise_error(o.float().cpu(), o_ref.double().cpu()) <= 2e-2
        assert orc.normwise_error(lse.cpu(), lse_ref.double().cpu()) <= 2e-2


def test_noalloc_rejects_problems_beyond_its_scratch():
    base = workloads.WORKLOADS[1]
    dev = torch.device("cuda")
    lay = api.pack([4096], [8], [512] * 8, dev)      # rotated Q + K need 64 MiB > 16 MiB
    T = lay.total_tokens
    q = torch.zeros((T, 32, 128), dtype=torch.bfloat16, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty((32, T), dtype=torch.float32, device=dev)
    st = call_noalloc(lay, q, q, q, o, lse, base.rope_theta)
    assert st == _lib.PG_ERR_INVALID_ARG
    assert b"scratch" in _lib.lib().pg_last_error_message()
