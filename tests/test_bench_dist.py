"""The multi-rank path of bench.py on CPU: two gloo ranks, no GPU.

Each rank runs its own copy of the workload (weak scaling; nothing is
exchanged on the data path), so the only cross-rank logic is the rendezvous
and the max over ranks of the timed region, which is what this checks.
"""

import os
import socket

import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench
    r, w, local = bench.dist_setup(world)
    got = bench.barrier_max(10.0 + 5.0 * r, w)
    out.put((r, w, local, got))
    import torch.distributed as dist
    dist.destroy_process_group()



def test_two_gloo_ranks_take_the_max_of_the_timed_region():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == [(0, 2, 0, 15.0), (1, 2, 1, 15.0)]


def test_flop_count_matches_the_pair_formula():
    import bench
    from scaled_dot_product_07_gb300 import workloads as W
    w = W.WORKLOADS["decoder_long"]
    assert bench.pairs(w) == 4096 * 4097 // 2
    f, b = bench.flops(w)
    assert f == 4 * 128 * 8390656 * 128 and b == 2.5 * f
    c = W.WORKLOADS["cross_attn"]
    assert bench.pairs(c) == 1024 * 8192
    # causal with more queries than keys: rows past Sk see every key
    w2 = W.make_workload("tiny", Sq=10, Sk=4)
    assert bench.pairs(w2) == sum(min(i + 1, 4) for i in range(10))


def test_small_kernel_bytes_of_the_backward():
    """Bytes behind the HBM roofline of the backward's preprocess and dQ
    conversion: at B8 H16 S4096 D128, 0.543 GB (out, dout read; lse read;
    lse2, Delta and the zeroed 128-column fp32 accumulator written) plus
    0.403 GB (accumulator read, dq written)."""
    import bench
    from scaled_dot_product_07_gb300 import workloads as W
    w = W.WORKLOADS["decoder_long"]
    heads, rows = 8 * 16, 4096
    out_dout = 2 * rows * 128 * 2          # bf16 rows of out and dout
    written = rows * (128 + 2) * 4         # accumulator zeros, lse2, Delta
    convert = rows * 128 * 4 + rows * 128 * 2
    assert bench.bwd_small_kernel_bytes(w) == heads * (out_dout + 4 * rows + written + convert)
    # a smaller head dim reads and writes only its own columns, but the
    # accumulator rows stay 128 wide; Sq is padded to 128 for the written rows
    w64 = W.make_workload("tiny", Sq=200, D=64)
    pad = 256
    per_head = 2 * 200 * 64 * 2 + 4 * 200 + pad * 130 * 4 + 200 * 64 * 6
    assert bench.bwd_small_kernel_bytes(w64) == w64.B * w64.H * per_head
