"""N > 1 path on the CPU: two gloo ranks own disjoint (batch, kv-group) units
of one problem, compute their units' forward and backward with no exchange,
and the gathered results equal the single-process result.  (The GPU
benchmark uses the same sharding with one GPU per rank; collectives there
carry only timing.)"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from exact_attention_85_gb300.sharding import query_heads, unit_range, units

B, Hq, Hkv, N, d = 3, 4, 2, 24, 8


def _inputs():
    g = torch.Generator().manual_seed(5)
    q = torch.randn(B, Hq, N, d, generator=g, dtype=torch.float64)
    k = torch.randn(B, Hkv, N, d, generator=g, dtype=torch.float64)
    v = torch.randn(B, Hkv, N, d, generator=g, dtype=torch.float64)
    dO = torch.randn(B, Hq, N, d, generator=g, dtype=torch.float64)
    return q, k, v, dO


def _worker(rank, world, port, out_dir):
    import oracle
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    q, k, v, dO = _inputs()
    o = torch.zeros(B, Hq, N, d, dtype=torch.float64)
    dq = torch.zeros_like(q)
    dk = torch.zeros_like(k)
    dv = torch.zeros_like(v)
    for b, g in units(B, Hkv, world, rank):
        hs = list(query_heads(g, Hq, Hkv))
        # a unit's data only: its query heads and its key/value head
        qs, ks, vs, dOs = (t[b:b + 1, sl] for t, sl in ((q, hs), (k, [g]), (v, [g]), (dO, hs)))
        ou, _ = oracle.attention_fwd(qs, ks, vs, True, 0.3)
        gq, gk, gv = oracle.attention_bwd(qs, ks, vs, dOs, True, 0.3)
        o[b, hs] = torch.from_numpy(ou[0])
        dq[b, hs] = torch.from_numpy(gq[0])
        dk[b, g] = torch.from_numpy(gk[0, 0])
        dv[b, g] = torch.from_numpy(gv[0, 0])
    # gather only to check the result (not part of the sharded computation)
    outs = []
    for t in (o, dq, dk, dv):
        parts = [torch.zeros_like(t) for _ in range(world)]
        dist.all_gather(parts, t)
        outs.append(sum(parts))
    lo, hi = unit_range(B, Hkv, world, rank)
    spans = [torch.zeros(2, dtype=torch.int64) for _ in range(world)]
    dist.all_gather(spans, torch.tensor([lo, hi]))
    if rank == 0:
        torch.save({"outs": outs, "spans": [s.tolist() for s in spans]}, os.path.join(out_dir, "res.pt"))
    dist.barrier()
    dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_unit_partition_is_disjoint_and_complete():
    for total_b, hkv, world in ((3, 2, 2), (4, 8, 3), (1, 1, 4), (5, 3, 7)):
        seen = []
        for r in range(world):
            lo, hi = unit_range(total_b, hkv, world, r)
            assert 0 <= lo <= hi <= total_b * hkv
            seen += list(range(lo, hi))
        assert seen == list(range(total_b * hkv))
    with pytest.raises(ValueError):
        unit_range(2, 2, 2, 2)


def test_two_gloo_ranks_match_single_process(tmp_path):
    import oracle
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, start_method="spawn")
    res = torch.load(os.path.join(tmp_path, "res.pt"))
    assert res["spans"] == [[0, 3], [3, 6]]
    q, k, v, dO = _inputs()
    o_ref, _ = oracle.attention_fwd(q, k, v, True, 0.3)
    rq, rk, rv = oracle.attention_bwd(q, k, v, dO, True, 0.3)
    for got, ref in zip(res["outs"], (o_ref, rq, rk, rv)):
        np.testing.assert_allclose(got.numpy(), ref, atol=1e-12)


# ----------------------------------------------- packed variable-length batch

LENGTHS = [7, 0, 30, 3, 12, 25, 1]
HQ_V, HKV_V, D_V = 4, 2, 8


def _varlen_inputs():
    g = torch.Generator().manual_seed(9)
    total = sum(LENGTHS)
    q = torch.randn(total, HQ_V, D_V, generator=g, dtype=torch.float64)
    k = torch.randn(total, HKV_V, D_V, generator=g, dtype=torch.float64)
    v = torch.randn(total, HKV_V, D_V, generator=g, dtype=torch.float64)
    dO = torch.randn(total, HQ_V, D_V, generator=g, dtype=torch.float64)
    cu = np.concatenate([[0], np.cumsum(LENGTHS)])
    return q, k, v, dO, cu


def _varlen_worker(rank, world, port, out_dir):
    import oracle
    from exact_attention_85_gb300.sharding import varlen_shard
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    q, k, v, dO, cu = _varlen_inputs()
    _, _, r0, r1, lcu = varlen_shard(cu, world, rank)
    outs = [torch.zeros_like(t) for t in (q, q, k, v)]
    if r1 > r0:
        # this rank's rows only, with offsets relative to its first row
        o, _ = oracle.attention_fwd_varlen(q[r0:r1], k[r0:r1], v[r0:r1], lcu, True, 0.4)
        gq, gk, gv = oracle.attention_bwd_varlen(q[r0:r1], k[r0:r1], v[r0:r1], dO[r0:r1], lcu, True, 0.4)
        for t, val in zip(outs, (o, gq, gk, gv)):
            t[r0:r1] = torch.from_numpy(val)
    gathered = []
    for t in outs:
        parts = [torch.zeros_like(t) for _ in range(world)]
        dist.all_gather(parts, t)
        gathered.append(sum(parts))
    if rank == 0:
        torch.save(gathered, os.path.join(out_dir, "varlen.pt"))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_packed_batch_without_exchange(tmp_path):
    import oracle
    port = _free_port()
    mp.spawn(_varlen_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    got = torch.load(os.path.join(tmp_path, "varlen.pt"))
    q, k, v, dO, cu = _varlen_inputs()
    ro, _ = oracle.attention_fwd_varlen(q, k, v, cu, True, 0.4)
    rq, rk, rv = oracle.attention_bwd_varlen(q, k, v, dO, cu, True, 0.4)
    for t, ref in zip(got, (ro, rq, rk, rv)):
        np.testing.assert_allclose(t.numpy(), ref, atol=1e-12)


def test_varlen_shard_balances_and_covers():
    from exact_attention_85_gb300.sharding import varlen_shard
    cu = [0, 5, 5, 6, 15, 19, 1000, 1010]
    for world in (1, 2, 3, 5):
        spans = [varlen_shard(cu, world, r) for r in range(world)]
        assert spans[0][0] == 0 and spans[-1][1] == len(cu) - 1
        for a, b in zip(spans, spans[1:]):
            assert a[1] == b[0] and a[3] == b[2]  # contiguous, no gaps or overlaps
        for lo, hi, r0, r1, lcu in spans:
            assert lcu == [c - r0 for c in cu[lo:hi + 1]] and r1 - r0 == lcu[-1]
    # the long sequence gets a rank of its own
    assert varlen_shard(cu, 2, 1)[:2] == (5, 7) or varlen_shard(cu, 2, 1)[:2] == (6, 7)
