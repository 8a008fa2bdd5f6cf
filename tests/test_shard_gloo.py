"""The vocabulary-sharded verify's exchange between ranks, world size 2 over gloo (CPU).

Each rank holds columns [v0, v1) of the same seeded rows (shard.shard_bounds)
and writes one record per row in the library's record format (sv.h,
sv_shard_record_bytes: status, count, then the top-32 composite keys --
logit order key above, whole-vocabulary index inverted below -- descending).
The records here are made on the host (the library's producer is a GPU
kernel); what is checked is the exchange the library leaves to the caller:
shard.exchange_records gathers equal-sized buffers from both ranks, after
which each rank's merge of the gathered records gives the top k of the whole
rows -- the same keys, in the same order, with the lowest index first among
equal logits -- and the oracle's argmax and kept set.
"""
import os
import socket

import numpy as np
import torch.multiprocessing as mp

RECORD = 264   # bytes: uint32 status, uint32 count, 32 x uint64 keys


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _order_key(v):
    b = np.asarray(v, np.float32).view(np.uint32).astype(np.uint64)
    b = np.where((b & 0x7FFFFFFF) == 0, np.uint64(0), b)
    return np.where(b & 0x80000000, ~b & 0xFFFFFFFF, b | 0x80000000).astype(np.uint64)


def _keys(vals, idx):
    return (_order_key(vals) << np.uint64(32)) | (np.uint64(0xFFFFFFFF) - idx.astype(np.uint64))


def _rows(seed=11, rows=6, V=1003):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((rows, V)) * 3).astype(np.float32)
    x[:, 5] = x[:, 900] = x.max(axis=1) + 1.0    # ties across the shard boundary: lower index first
    x[2, :] = np.float32(0.5)                    # a row of equal values
    return x


def _records(x, v0, v1, k):
    out = np.zeros((x.shape[0], RECORD), np.uint8)
    for r in range(x.shape[0]):
        idx = np.arange(v0, v1)
        keys = np.sort(_keys(x[r, v0:v1], idx))[::-1][:k]
        rec = out[r]
        rec[0:4] = np.frombuffer(np.uint32(0).tobytes(), np.uint8)
        rec[4:8] = np.frombuffer(np.uint32(len(keys)).tobytes(), np.uint8)
        rec[8:8 + 8 * len(keys)] = np.frombuffer(keys.astype(np.uint64).tobytes(), np.uint8)
    return out


def _merge(gathered, k):
    world, rows, _ = gathered.shape
    merged = []
    for r in range(rows):
        ks = []
        for s in range(world):
            rec = gathered[s, r]
            cnt = int(np.frombuffer(rec[4:8].tobytes(), np.uint32)[0])
            ks.extend(np.frombuffer(rec[8:8 + 8 * cnt].tobytes(), np.uint64).tolist())
        merged.append(sorted(ks, reverse=True)[:k])
    return merged


def _worker(rank, world, port, q, k):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch
    import torch.distributed as dist
    from speculative_decoding_verification_rows_gb300 import shard
    dist.init_process_group("gloo", rank=rank, world_size=world)
    x = _rows()
    v0, v1 = shard.shard_bounds(x.shape[1], world, rank)
    mine = torch.from_numpy(_records(x, v0, v1, k).reshape(-1))
    got = shard.exchange_records(mine).numpy().reshape(world, x.shape[0], RECORD)
    q.put((rank, _merge(got, k)))
    dist.destroy_process_group()


def test_two_ranks_exchange_then_merge_give_the_whole_rows_top_k():
    import oracle
    k = 20
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q, k)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=5) for _ in range(2))
    assert res[0] == res[1]                      # every rank merges to the same records
    x = _rows()
    for r in range(x.shape[0]):
        whole = sorted(_keys(x[r], np.arange(x.shape[1])).tolist(), reverse=True)[:k]
        assert res[0][r] == whole
        # the oracle's argmax and top-k set (T = 1, top-k 20, no top-p) from the merged keys
        d, probs = oracle.row_transform(x[r], 1.0, k, 1.0)
        top_idx = [0xFFFFFFFF - (key & 0xFFFFFFFF) for key in res[0][r]]
        assert top_idx[0] == d["argmax"]
        assert sorted(top_idx) == sorted(np.nonzero(probs > 0)[0].tolist())


def test_shard_bounds_cover_the_vocabulary():
    from speculative_decoding_verification_rows_gb300 import shard
    for V in (4, 7, 1003, 248_320):
        for world in range(1, 5):
            if world > V:
                continue
            b = [shard.shard_bounds(V, world, r) for r in range(world)]
            assert b[0][0] == 0 and b[-1][1] == V
            assert all(b[i][1] == b[i + 1][0] for i in range(world - 1))
            assert max(v1 - v0 for v0, v1 in b) - min(v1 - v0 for v0, v1 in b) <= 1
