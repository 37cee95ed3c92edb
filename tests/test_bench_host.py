"""Host-side checks of bench.py's bookkeeping: pair counts, byte counts and the
multi-rank aggregation (world size 2 over gloo on the CPU)."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

import bench
import numpy as np
import oracle


@pytest.mark.parametrize("Sq,Sk,mode,w,g", [(37, 37, 0, 0, 0), (37, 37, 1, 0, 0),
                                            (20, 45, 1, 0, 0), (45, 20, 1, 0, 0),
                                            (200, 200, 2, 16, 5), (100, 130, 2, 7, 40),
                                            (64, 64, 2, 1, 0), (64, 64, 2, 100, 100),
                                            (90, 90, 3, 0, 0), (90, 90, 3, 7, 0),
                                            (40, 100, 3, 13, 0), (100, 40, 3, 13, 0),
                                            (64, 64, 3, 1000, 0), (90, 90, 4, 0, 0),
                                            (90, 90, 4, 0, 30), (40, 100, 4, 0, 70),
                                            (100, 40, 4, 0, 20), (64, 64, 4, 0, 500)])
def test_visible_pairs_matches_oracle_count(Sq, Sk, mode, w, g):
    assert bench.visible_pairs(Sq, Sk, mode, w, g) == oracle.count_visible(Sq, Sk, mode, w, g)


def test_headline_flop_counts():
    assert bench.prefill_flops(bench.PREFILL["causal4k"]) == 4 * 128 * 128 * 8_390_656
    assert bench.prefill_flops(bench.PREFILL["noncausal4k"]) == 4 * 128 * 128 * 4096 * 4096
    assert bench.prefill_flops(bench.PREFILL["causal2k"]) == 4 * 128 * 128 * 2_098_176
    assert bench.prefill_flops(bench.PREFILL["window32k"]) == 4 * 32 * 128 * 66_976_800
    # band +-512 over 4096 rows: 3072 interior rows of 1025 keys, 2 x 512 edge rows
    # of 513..1024 keys
    assert bench.prefill_flops(bench.PREFILL["band4k"]) == 4 * 128 * 128 * (
        3072 * 1025 + 2 * (512 * 513 + 511 * 512 // 2))
    # prefix 1024: the first 1024 rows see 1024 keys, row i >= 1024 sees i + 1
    assert bench.prefill_flops(bench.PREFILL["prefixlm4k"]) == 4 * 128 * 128 * (
        1024 * 1024 + 4096 * 4097 // 2 - 1024 * 1025 // 2)


def test_decode_bytes():
    # 16384 bytes per context token (K and V, 32 heads x 128 x 2 bytes) plus q, o, lse, tables
    assert bench.decode_bytes([1, 2], 2, 32, 128, 32) == 3 * 16384 + 2 * 2 * 32 * 128 * 2 \
        + 2 * 32 * 4 + 2 * 32 * 4 + 2 * 4


def _worker(rank, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE="2", LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=2)
    t = bench.max_over_ranks(1.5 + rank, 2)
    v = bench.aggregate(100.0, t, 2)
    bench.barrier(2)
    out[rank] = (t, v)
    dist.destroy_process_group()


def test_two_rank_aggregation_over_gloo():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    procs = [ctx.Process(target=_worker, args=(r, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(2):
        t, v = out[r]
        assert t == 2.5                      # the slowest rank's time
        assert v == pytest.approx(200.0 / 2.5)  # both ranks' units over that time


@pytest.mark.parametrize("H,Sq,Sk,blk", [(2, 300, 300, 128), (3, 130, 257, 128), (1, 9, 7, 4)])
def test_layout_pairs_match_oracle_count(H, Sq, Sk, blk):
    from tiled_attention_06_gb300 import inputs
    lay = inputs.block_layout(H, Sq, Sk, block=blk, seed=H + Sq)
    assert bench.layout_pairs(lay, Sq, Sk, blk) == oracle.count_visible_layout(H, Sq, Sk,
                                                                             lay.numpy(), blk)


def test_bigbird_layout_shape():
    from tiled_attention_06_gb300 import inputs
    lay = inputs.block_layout(4, 4096, 4096, seed=0).numpy()
    assert lay.shape == (4, 32, 32) and lay.dtype == np.uint8
    i, j = np.indices((32, 32))
    assert np.all(lay[:, np.abs(i - j) <= 1] == 1)       # local band
    assert np.all(lay[:, 0, :] == 1) and np.all(lay[:, :, 0] == 1)  # global block
    assert np.all(lay[:, 1:].sum(-1) <= 3 + 1 + 2)       # band, global column, two random


def test_captured_traffic_only_for_its_workloads():
    """A captured DRAM figure is reported only for the workloads it was taken on (and only
    while the kernel sources hash as captured); an explicit figure always wins."""
    for kind, t in bench.NCU_TRAFFIC.items():
        current = t["bytes"] is not None and t["sha256"] == bench.sources_sha(t["sources"])
        for w in t["workloads"]:
            assert bench.ncu_traffic(kind, w, None) == (t["bytes"] if current else None)
        for w in ("band4k", "blocksparse4k", "window32k", None):
            assert w in t["workloads"] or bench.ncu_traffic(kind, w, None) is None
        assert bench.ncu_traffic(kind, "band4k", 123.0) == 123.0
