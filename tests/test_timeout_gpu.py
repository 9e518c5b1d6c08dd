"""Kernel-side failure detection without a GPU fault: a debug flag makes the tensor-core forward
withhold the 'P ready' signal, so its bounded waits run out; the kernel must record
PG_ERR_TIMEOUT in the status word, exit cleanly (copies in flight awaited, TMEM freed), and leave
the context usable for the next call."""
import pytest
import torch

from oracle import prefix_grouper_oracle as orc
from shared_prefix_grouped_gb300 import _lib, api, workloads
from shared_prefix_grouped_gb300.build import build

pytestmark = pytest.mark.gpu

PG_DEBUG_WITHHOLD_P = 1


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build()


def test_withheld_signal_times_out_and_context_survives():
    w = workloads.small_variant(workloads.WORKLOADS[1], prefix_len=150, suffix_lens=[40, 60],
                                heads_q=1, heads_kv=1)
    prob = workloads.make_problem(w)
    dev = torch.device("cuda")
    lay = api.pack(prob.prefix_lens, prob.group_sizes, prob.suffix_lens, dev)
    q, k, v = (t.to(dev) for t in (prob.q, prob.k, prob.v))
    assert api.device_status() == 0
    api.grouped_attn_fwd(lay, q, k, v, rope_theta=w.rope_theta, debug=PG_DEBUG_WITHHOLD_P)
    torch.cuda.synchronize()
    assert api.device_status(clear=True) == _lib.PG_ERR_TIMEOUT
    assert api.device_status() == 0
    # the same call without the flag still works and is correct
    o, lse = api.grouped_attn_fwd(lay, q, k, v, rope_theta=w.rope_theta)
    torch.cuda.synchronize()
    assert api.device_status() == 0
    ref = orc.repeated_prefix(orc.pack_layout(prob.prefix_lens, prob.group_sizes,
                                              prob.suffix_lens), prob.q, prob.k, prob.v,
                              theta=w.rope_theta)
    assert orc.normwise_error(o.float().cpu(), ref.o) <= 2e-2
