"""Full-size equivalence on the GPU: grouped attention against the repeated-prefix layout (every
[P; Ri] materialised as its own sequence) run through the same kernels, for the three bf16
workloads, in the benchmark's launch configuration (one workspace per step, the forward's
rotation kept for the backward).

The abstract page of Prefix Grouper claims identical forward outputs and backward gradients for
the two computations; the Pith review ("What would settle it") asks for exactly this comparison
of outputs and gradients.  Mapping: O and LSE of each packed row from the copy that receives its
upstream gradient (prefix rows: the group's first copy), dQ / dK / dV summed over the copies.
Normwise tolerance 2e-2, the bf16 criterion.
"""
import argparse
import os
import sys

import pytest
import torch

from shared_prefix_grouped_gb300 import workloads
from shared_prefix_grouped_gb300.build import build

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build()


@pytest.mark.parametrize("wi", [1, 2, 3])
def test_grouped_equals_repeated_full_size(wi):
    w = workloads.WORKLOADS[wi]
    prob = workloads.make_problem(w)
    dev = torch.device("cuda")
    step = bench.Step(prob, dev)
    args = argparse.Namespace(steps=3)
    out = bench.repeated_leg(prob, dev, 0, 1.0, args, grouped=step)
    print(w.name, out["normwise_err"])
    assert out["max_normwise_err"] <= 2e-2, out["normwise_err"]
    del step
    torch.cuda.empty_cache()
