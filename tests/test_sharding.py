"""Multi-rank logic on CPU: world_size-2 gloo ranks each run the oracle on their shard; the
rank-ordered reduction of the prefix gradient reproduces the unsharded result."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from oracle import prefix_grouper_oracle as orc
from shared_prefix_grouped_gb300 import sharding


def free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def make_case():
    lp, rs = 9, [4, 7, 2, 5, 3]
    lay = orc.pack_layout([lp], [len(rs)], rs)
    g = torch.Generator().manual_seed(5)
    T, Hq, Hkv, d = lay.total_tokens, 4, 2, 8
    mk = lambda h: torch.randn((T, h, d), generator=g, dtype=torch.float64)
    return lp, rs, lay, mk(Hq), mk(Hkv), mk(Hkv), mk(Hq)


def rank_main(rank, world, port, out_path):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    lp, rs, lay, q, k, v, do = make_case()
    mine = sharding.split_responses(len(rs), world, rank)
    rows = sharding.shard_rows(lp, rs, mine)
    sub = orc.pack_layout([lp], [len(mine)], [rs[i] for i in mine])
    do_r = sharding.route_prefix_do(do[rows], lp, rank)
    res = orc.repeated_prefix(sub, q[rows], k[rows], v[rows], do_r, theta=20.0)
    pre = torch.cat([res.dq[:lp].flatten(), res.dk[:lp].flatten(), res.dv[:lp].flatten()])
    total = sharding.allgather_prefix_grads(pre)
    # gather the response rows' results too
    payload = {"rank": rank, "rows": rows[lp:], "o": res.o[lp:], "dq": res.dq[lp:],
               "dk": res.dk[lp:], "dv": res.dv[lp:], "prefix": total, "o_prefix": res.o[:lp]}
    objs = [None] * world
    dist.all_gather_object(objs, payload)
    if rank == 0:
        torch.save(objs, out_path)
    dist.destroy_process_group()


def test_two_rank_response_split_matches_unsharded(tmp_path):
    world = 2
    out = str(tmp_path / "gathered.pt")
    mp.start_processes(rank_main, args=(world, free_port(), out), nprocs=world, start_method="spawn")
    objs = torch.load(out, weights_only=False)
    lp, rs, lay, q, k, v, do = make_case()
    ref = orc.repeated_prefix(lay, q, k, v, do, theta=20.0)
    n = lp * 4 * 8
    m = lp * 2 * 8
    prefix = objs[0]["prefix"]
    assert torch.allclose(prefix[:n].view(lp, 4, 8), ref.dq[:lp], atol=1e-12)
    assert torch.allclose(prefix[n:n + m].view(lp, 2, 8), ref.dk[:lp], atol=1e-12)
    assert torch.allclose(prefix[n + m:].view(lp, 2, 8), ref.dv[:lp], atol=1e-12)
    # both ranks reduced to the identical (bitwise) prefix gradient
    assert torch.equal(objs[0]["prefix"], objs[1]["prefix"])
    for o in objs:
        rows = o["rows"]
        assert torch.allclose(o["o"], ref.o[rows], atol=1e-12)
        assert torch.allclose(o["dq"], ref.dq[rows], atol=1e-12)
        assert torch.allclose(o["dk"], ref.dk[rows], atol=1e-12)
        assert torch.allclose(o["o_prefix"], ref.o[:lp], atol=1e-12)


def test_group_assignment_balances_and_covers():
    plens = [2048] * 8
    gs = [16] * 8
    g = torch.Generator().manual_seed(1)
    rs = [int(x) for x in torch.randint(64, 513, (128,), generator=g)]
    for world in (1, 2, 3, 8):
        parts = sharding.assign_groups(plens, gs, rs, world)
        assert sorted(b for p in parts for b in p) == list(range(8))
    parts = sharding.assign_groups([100, 10, 10, 10], [1, 1, 1, 1], [0, 0, 0, 0], 2)
    assert parts == [[0], [1, 2, 3]]


def test_split_responses_partitions():
    for n in (0, 1, 5, 16):
        for world in (1, 2, 3, 4):
            got = [i for r in range(world) for i in sharding.split_responses(n, world, r)]
            assert got == list(range(n))
