"""The boundary used from plain C: tests/c/abi_from_c.c (C99, headers only from include/) is
compiled with gcc against the library, runs the host-side entry points (packing of the three
layouts, workspace sizes, an argument error) and prints them; every line must equal what the
Python binding gets from the same calls.  Needs no GPU."""
import os
import shutil
import subprocess

import pytest
import torch

from shared_prefix_grouped_gb300 import _lib, api
from shared_prefix_grouped_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def c_output(tmp_path_factory):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    build()
    libdir = os.path.dirname(_lib.LIB_PATH)
    exe = str(tmp_path_factory.mktemp("abi_c") / "abi_from_c")
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                    "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c",
                                                                      "abi_from_c.c"),
                    "-L", libdir, "-lpg_gb300", f"-Wl,-rpath,{libdir}", "-o", exe], check=True)
    out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout
    return {line.split(" ", 1)[0]: line.split(" ", 1)[1] for line in out.splitlines()}


def check_layout(c, name, pos, st):
    assert int(c[f"{name}_tokens"]) == st.total_tokens
    assert int(c[f"{name}_pairs"]) == st.pairs
    assert int(c[f"{name}_depth"]) == st.max_depth
    assert int(c[f"{name}_pad_rows"]) == st.n_pad_rows
    assert [int(x) for x in c[f"{name}_pos"].split()] == pos.tolist()


def test_packing_from_c_matches_the_binding(c_output):
    pos, _, st = api.pack_host([5, 0], [3, 2], [2, 0, 3, 4, 1])
    check_layout(c_output, "packed", pos, st)
    pos, _, st = api.pack_tree_host([-1, 0, 1, 1, 0], [2, 1, 2, 1, 1])
    check_layout(c_output, "tree", pos, st)
    pos, _, st = api.pack_padded_host(2, 5, 3, 4, [4, 0, 2, 1, 4, 3])
    check_layout(c_output, "padded", pos, st)


def test_workspace_and_errors_from_c_match_the_binding(c_output):
    pos, tab, st = api.pack_host([5, 0], [3, 2], [2, 0, 3, 4, 1])
    lay = api.Layout([5, 0], [3, 2], [2, 0, 3, 4, 1], st, pos, tab)
    for key, flags in [("ws_plain", 0), ("ws_pre", _lib.PG_FLAG_PRE_ROTATED)]:
        n = api.workspace_size(lay, torch.bfloat16, 4, 2, 128, api.make_opts(1e4, 0.0, flags), 1)
        assert int(c_output[key]) == n
    code, text = c_output["bad_heads"].split(" ", 1)
    assert int(code) == _lib.PG_ERR_INVALID_ARG
    assert text == _lib.lib().pg_status_string(_lib.PG_ERR_INVALID_ARG).decode()
