"""The counts exchange of sharded layers on two gloo ranks (CPU).

Each rank counts its own routes, exchange_counts (the binding's all-gather
over a torch.distributed group) stacks every rank's counts in rank order,
and from that table plus its own topk_idx a rank has what the sharded
prepare needs: every owner's expert offsets and its own routes' receive rows.
The rows derived here from the gathered table must equal the sharded
oracle's, computed from both ranks' full routing tables."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

N, E, K, A = 2, 8, 3, 4


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _idx(rank):
    from combine_ep_prepare_gb300 import workloads as wl
    idx, _ = wl.random_routing([37, 52][rank], K, E, seed=500 + rank, p_mask=0.1)
    return idx


def _rows_from_table(all_counts, idx, rank):
    """Receive rows of this rank's routes from the gathered counts: per owner,
    blocks of its experts padded to A; inside a block the routes of lower
    ranks first, then this rank's in (t, k) order."""
    tot = all_counts.sum(axis=0)
    el = E // N
    padded = (tot + A - 1) // A * A
    off = np.zeros(E, np.int64)
    for q in range(N):
        off[q * el:(q + 1) * el] = np.concatenate([[0], np.cumsum(padded[q * el:(q + 1) * el])[:-1]])
    nxt = off + all_counts[:rank].sum(axis=0)
    rows = np.full(idx.size, -1, np.int64)
    for i, e in enumerate(idx.reshape(-1)):
        if 0 <= e < E:
            rows[i] = nxt[e]
            nxt[e] += 1
    return rows.reshape(idx.shape), off


def _worker(rank, port, out):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import torch
    import torch.distributed as dist
    from combine_ep_prepare_gb300 import _libep
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=N)
    idx = _idx(rank).numpy()
    v = idx.reshape(-1)
    local = torch.from_numpy(np.bincount(v[(v >= 0) & (v < E)], minlength=E).astype(np.int32))
    table = _libep.exchange_counts(local)
    rows, off = _rows_from_table(table.numpy(), idx, rank)
    out[rank] = (table.numpy().tolist(), rows.tolist(), off.tolist())
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_counts_exchange(oracle_mod):
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, port, out)) for r in range(N)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(180)
        assert p.exitcode == 0
    idx = [_idx(r).numpy() for r in range(N)]
    sr = oracle_mod.shard_prepare(idx, E, A, N)
    for r in range(N):
        table, rows, off = out[r]
        assert table == out[0][0]  # every rank holds the same table, rows in rank order
        v = idx[r].reshape(-1)
        assert table[r] == np.bincount(v[(v >= 0) & (v < E)], minlength=E).tolist()
        assert np.array_equal(np.array(rows), sr.slot[r])
        assert off == sr.offsets[:E].tolist()


def _rm_rows_from_table(all_counts, idx, rank):
    """Rank-major rows of this rank's tokens from the gathered per-owner
    counts: on owner q, the tokens of lower ranks first, then this rank's in
    token order; every route of a token to q shares its row."""
    el = E // N
    nxt = all_counts[:rank].sum(axis=0).astype(np.int64)
    rows = np.full(idx.shape, -1, np.int64)
    for t, toks in enumerate(idx):
        row_of = {}
        for k, e in enumerate(toks):
            if 0 <= e < E:
                q = int(e // el)
                if q not in row_of:
                    row_of[q] = nxt[q]
                    nxt[q] += 1
                rows[t, k] = row_of[q]
    return rows


def _rm_worker(rank, port, out):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import torch
    import torch.distributed as dist
    from combine_ep_prepare_gb300 import _libep
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=N)
    idx = _idx(rank).numpy()
    el = E // N
    goes = np.zeros(N, np.int32)
    for toks in idx:
        goes += np.isin(np.arange(N), [int(e // el) for e in toks if 0 <= e < E]).astype(np.int32)
    table = _libep.exchange_counts(torch.from_numpy(goes))
    out[rank] = (table.numpy().tolist(), _rm_rows_from_table(table.numpy(), idx, rank).tolist())
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_rank_major_counts_exchange(oracle_mod):
    """Rank-major layers exchange [N] counts per rank (tokens per owner);
    the gathered [N][N] table gives every rank its rows on every owner, equal
    to the rank-major oracle's."""
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rm_worker, args=(r, port, out)) for r in range(N)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(180)
        assert p.exitcode == 0
    idx = [_idx(r).numpy() for r in range(N)]
    rr = oracle_mod.rm_prepare(idx, E, N)
    for r in range(N):
        table, rows = out[r]
        assert table == out[0][0] == rr.counts.tolist()
        assert np.array_equal(np.array(rows), rr.row[r])
