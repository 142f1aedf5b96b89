"""World-size-2 gloo tests on CPU of the multi-rank logic (no GPU):

* the bench's barrier and max-over-ranks timing plumbing;
* the sharding invariants a multi-GPU layout would rely on, checked with the
  oracle: 1x128 quantization commutes with 128-aligned token sharding (an
  all_gather of per-rank quantizations equals the full one), and a K-sharded
  ("rowwise" tensor-parallel) forward GEMM summed by all_reduce equals the
  unsharded product, because 128-aligned K shards keep every scale block local.
"""
import os
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, fn_name, q):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q.put((rank, globals()[fn_name](rank, world)))
    except Exception as e:  # report, never hang the parent
        q.put((rank, repr(e)))
    finally:
        dist.destroy_process_group()


def _run(fn_name, world=2):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + (os.getpid() % 2000)
    procs = [ctx.Process(target=_worker, args=(r, world, port, fn_name, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
    return out


def _bench_plumbing(rank, world):
    import bench
    bench.barrier(world)
    return bench.max_over_ranks(world, 1.5 + rank, "cpu")


def _quant_sharding(rank, world):
    import oracle
    from mxfp8_precision_gemms_fp8bw_gb300 import inputs
    t = inputs.tiny()
    x = inputs.bf16_to_f32_numpy(t.x)                     # [256, 512]
    rows = x.shape[0] // world
    q, s = oracle.quant_1x128_row(np.ascontiguousarray(x[rank * rows:(rank + 1) * rows]))
    gq = [torch.empty((rows, x.shape[1]), dtype=torch.uint8) for _ in range(world)]
    gs = [torch.empty(s.shape, dtype=torch.float32) for _ in range(world)]
    dist.all_gather(gq, torch.from_numpy(q))
    dist.all_gather(gs, torch.from_numpy(s))
    fq, fs = oracle.quant_1x128_row(x)
    return bool(np.array_equal(torch.cat(gq).numpy(), fq) and np.array_equal(torch.cat(gs, 1).numpy(), fs))


def _rowwise_tp(rank, world):
    import oracle
    from mxfp8_precision_gemms_fp8bw_gb300 import inputs
    t = inputs.tiny()
    x, w = inputs.bf16_to_f32_numpy(t.x), inputs.bf16_to_f32_numpy(t.w)   # K = 512 split in two
    k = x.shape[1] // world
    xs, ws = np.ascontiguousarray(x[:, rank * k:(rank + 1) * k]), np.ascontiguousarray(w[:, rank * k:(rank + 1) * k])
    xq, xsc = oracle.quant_1x128_row(xs)
    wq, _, wsc = oracle.quant_128x128(ws)
    part = torch.from_numpy(oracle.gemm_fwd(xq, xsc, wq, wsc))
    dist.all_reduce(part)
    fq, fs = oracle.quant_1x128_row(x)
    wfq, _, wfs = oracle.quant_128x128(w)
    full = oracle.gemm_fwd(fq, fs, wfq, wfs)
    return float(np.max(np.abs(part.numpy() - full)) / np.max(np.abs(full)))


def test_bench_plumbing_two_ranks():
    out = _run("_bench_plumbing")
    assert out == {0: 2.5, 1: 2.5}


def test_token_sharded_quantization_equals_full():
    out = _run("_quant_sharding")
    assert out == {0: True, 1: True}


def test_k_sharded_forward_sums_to_full():
    out = _run("_rowwise_tp")
    assert all(isinstance(v, float) and v < 1e-12 for v in out.values()), out
