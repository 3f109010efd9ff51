"""Host-only ownership planner (muon_plan_assign): greedy cost balance of
whole matrices over data-parallel replicas.

Pinned against mathematics, not against itself: every member gets exactly one
rank; the list-scheduling bound (busiest rank <= total/R + (1 - 1/R) * largest
member); on small cases the optimum found by brute force over every
assignment, with Graham's longest-processing-time-first bound (<= (4/3 -
1/(3R)) times that optimum); equal members spread evenly; experts of a 3-D
parameter assigned one by one; the result is a function of its inputs only,
so two gloo ranks that run it on their own agree and partition the members.
"""
import itertools
import math

import pytest

import newton_schulz_bucket_gb300 as pkg
from newton_schulz_bucket_gb300 import _capi

MIXED = [[24, 10240]] * 5 + [[4, 512, 512]] + [[2048, 2048]] * 3 + [[4096, 1024], [1024, 4096]]


def test_every_member_owned_once_and_costs_add_up():
    r = pkg.assign_owners(MIXED, 4)
    assert len(r["owner"]) == len(r["members"]) == 5 + 4 + 3 + 2
    assert all(0 <= o < 4 for o in r["owner"])
    for rank in range(4):
        s = sum(c for c, o in zip(r["member_cost"], r["owner"]) if o == rank)
        assert math.isclose(s, r["rank_cost"][rank], rel_tol=1e-12)


@pytest.mark.parametrize("n_ranks", [1, 2, 3, 8, 64])
def test_list_scheduling_bound(n_ranks):
    # greedy list scheduling places each member on the least-loaded rank, so
    # the busiest rank ends below total / R + (1 - 1/R) * (largest member)
    r = pkg.assign_owners(MIXED, n_ranks)
    c = r["member_cost"]
    assert max(r["rank_cost"]) <= (sum(c) / n_ranks + (1 - 1 / n_ranks) * max(c)) * (1 + 1e-12)


def test_brute_force_small_cases():
    shapes = [[24, 10240], [2048, 2048], [2, 512, 1536], [1024, 1024], [3, 40, 640]]
    for n_ranks in (2, 3):
        r = pkg.assign_owners(shapes, n_ranks)
        c = r["member_cost"]
        best = min(max(sum(ci for ci, a in zip(c, assign) if a == k) for k in range(n_ranks))
                   for assign in itertools.product(range(n_ranks), repeat=len(c)))
        got = max(r["rank_cost"])
        assert got >= best * (1 - 1e-12)
        assert got <= (4 / 3 - 1 / (3 * n_ranks)) * best * (1 + 1e-12)


def test_equal_members_spread_evenly():
    # the pages' fused batch: 74 parameters of one shape over 8 replicas
    r = pkg.assign_owners([[24, 10240]] * 74, 8)
    counts = [r["owner"].count(k) for k in range(8)]
    assert sorted(counts) == [9] * 6 + [10] * 2
    assert counts == [10, 10, 9, 9, 9, 9, 9, 9]  # ties go to the lowest rank


def test_experts_assigned_individually():
    r = pkg.assign_owners([[8, 2048, 2048]], 4)
    assert [e for _, e in r["members"]] == list(range(8))
    assert sorted(r["owner"].count(k) for k in range(4)) == [2, 2, 2, 2]


def test_deterministic_and_cost_depends_on_path():
    a = pkg.assign_owners(MIXED, 5)
    b = pkg.assign_owners(MIXED, 5)
    assert a == b
    # a skinny member costs its memory traffic; a square one its tensor work
    r = pkg.assign_owners([[24, 10240], [4096, 4096]], 2)
    assert r["member_cost"][1] > 100 * r["member_cost"][0]


def test_bad_arguments_are_statuses():
    L = _capi.load()
    with pytest.raises(pkg.MuonError):
        pkg.assign_owners(MIXED, 0)
    with pytest.raises(pkg.MuonError):
        pkg.assign_owners(MIXED, 4, ns_steps=-1)
    sh = pkg._shapes(MIXED)
    o = pkg._options()
    assert L.muon_plan_assign(sh, len(MIXED), o, 5, 4, None, 0, None, None) == _capi.MUON_ERR_INVALID_ARG


def _assign_rank(rank, port, q):
    import os
    import sys
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import torch
    import torch.distributed as dist
    import newton_schulz_bucket_gb300 as p
    from newton_schulz_bucket_gb300 import workloads as W
    dist.init_process_group("gloo", rank=rank, world_size=2)
    r = p.assign_owners(W.get("c5_mixed_1000").shapes, 2)
    mine = torch.tensor([i for i, o in enumerate(r["owner"]) if o == rank], dtype=torch.int64)
    owners = torch.tensor(r["owner"], dtype=torch.int64)
    got = [torch.zeros_like(owners) for _ in range(2)]
    dist.all_gather(got, owners)
    n = torch.tensor([mine.numel()], dtype=torch.int64)
    counts = [torch.zeros_like(n) for _ in range(2)]
    dist.all_gather(counts, n)
    dist.destroy_process_group()
    q.put((rank, bool(torch.equal(got[0], got[1])), mine.tolist(), [int(c) for c in counts],
           len(r["owner"])))


def test_two_gloo_ranks_agree_on_owners():
    """Each replica runs the planner on its own; with no exchange of the
    result they must agree, and their owned sets must partition the members."""
    import multiprocessing as mp
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_assign_rank, args=(r, port, q)) for r in range(2)]
    for pr in procs:
        pr.start()
    for pr in procs:
        pr.join(timeout=120)
    for pr in procs:
        if pr.is_alive():
            pr.kill()
    assert all(pr.exitcode == 0 for pr in procs)
    res = sorted(q.get(timeout=5) for _ in range(2))
    assert all(agree for _, agree, _, _, _ in res)
    n = res[0][4]
    assert n == 1000
    owned = res[0][2] + res[1][2]
    assert sorted(owned) == list(range(n))
    assert res[0][3] == [len(res[0][2]), len(res[1][2])]
