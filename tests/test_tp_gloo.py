"""The tensor-parallel split of the MLP (nvfp4_quantized_dense_gb300.tp) on
the CPU: two gloo ranks each run their shard of the chain on the oracle,
all-reduce their fp32 partial down_proj outputs, and must match the
unsharded oracle -- h bit for bit on each rank's features, the output within
the GEMM tolerance.  Not run on more than one GPU."""
import os
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _setup(hid, inter, m):
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import oracle
    import synth
    x = synth.random_matrix((m, hid), (31, m, hid), scale=1.0)
    _, x = synth.to_bf16_bits(x)
    wgu = synth.random_matrix((2 * inter, hid), (32, inter, hid), scale=0.02)
    wdn = synth.random_matrix((hid, inter), (33, inter, hid), scale=0.02)
    gs_x = oracle.global_scale(np.abs(x).max())
    gs_gu, gs_dn = oracle.global_scale(np.abs(wgu).max()), oracle.global_scale(np.abs(wdn).max())
    gu, dn = oracle.quantize_nvfp4(wgu, gs_gu), oracle.quantize_nvfp4(wdn, gs_dn)
    xq, xs = oracle.quantize_nvfp4(x, gs_x)
    a_gu = np.float32(1.0) / (gs_x * gs_gu)
    h = oracle.swiglu_h(oracle.gemm_w4a4(xq, xs, gu[0], gu[1], a_gu, round_bf16=False))
    gs_h = oracle.global_scale(np.abs(h).max())
    a_dn = np.float32(1.0) / (gs_h * gs_dn)
    return oracle, x, gs_x, gu, dn, a_gu, gs_h, a_dn


def _worker(rank, world, port, shape, out):
    from nvfp4_quantized_dense_gb300 import tp
    hid, inter, m = shape
    oracle, x, gs_x, gu, dn, a_gu, gs_h, a_dn = _setup(hid, inter, m)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        f0, f1 = tp.shard_features(inter, world)[rank]
        xq, xs = oracle.quantize_nvfp4(x, gs_x)
        gq, gs = tp.shard_gate_up(gu[0], gu[1], inter, f0, f1)
        h_r = oracle.swiglu_h(oracle.gemm_w4a4(xq, xs, gq, gs, a_gu, round_bf16=False))
        hq_r, hs_r = oracle.quantize_nvfp4(h_r, gs_h)            # the shared static scale
        dq, ds = tp.shard_down(dn[0], dn[1], f0, f1)
        part = oracle.gemm_w4a4(hq_r, hs_r, dq, ds, a_dn, round_bf16=False).astype(np.float32)
        t = torch.from_numpy(part)
        dist.all_reduce(t, op=dist.ReduceOp.SUM)                 # the one exchange
        out[rank] = dict(f0=f0, f1=f1, hq=hq_r, hs=hs_r,
                         out=oracle.bf16_round(t.numpy().astype(np.float64)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("shape", [(256, 512, 4), (384, 1088, 5)])
def test_two_rank_tensor_parallel_mlp_matches_unsharded(shape):
    hid, inter, m = shape
    port = 29600 + (os.getpid() + inter) % 1000
    with mp.get_context("spawn").Manager() as mgr:
        res = mgr.dict()
        mp.start_processes(_worker, args=(2, port, shape, res), nprocs=2, join=True, start_method="spawn")
        res = dict(res)
    oracle, x, gs_x, gu, dn, a_gu, gs_h, a_dn = _setup(hid, inter, m)
    from tolerance import assert_gemm_close
    ref = oracle.mlp_w4a4_fused(x, gs_x, gu, a_gu, gs_h, dn, a_dn)
    xq, xs = oracle.quantize_nvfp4(x, gs_x)
    hq, hs = oracle.quantize_nvfp4(oracle.swiglu_h(oracle.gemm_w4a4(xq, xs, gu[0], gu[1], a_gu, round_bf16=False)),
                                   gs_h)
    assert [(res[r]["f0"], res[r]["f1"]) for r in (0, 1)] == [(0, res[1]["f0"]), (res[0]["f1"], inter)]
    for r in (0, 1):
        f0, f1 = res[r]["f0"], res[r]["f1"]
        assert (f1 - f0) % 64 == 0
        assert np.array_equal(res[r]["hq"], hq[:, f0 // 2:f1 // 2]), "rank's h codes differ from the unsharded h"
        assert np.array_equal(res[r]["hs"], hs[:, f0 // 16:f1 // 16]), "rank's h scales differ"
        assert_gemm_close(res[r]["out"], ref, what=f"rank {r} all-reduced output")
    assert np.array_equal(res[0]["out"], res[1]["out"])


def test_shard_plan_covers_whole_groups():
    sys.path.insert(0, ROOT)
    from nvfp4_quantized_dense_gb300 import tp
    for inter, world in [(17408, 2), (18432, 4), (18432, 8), (1088, 2), (64 * 7, 3)]:
        sh = tp.shard_features(inter, world)
        assert sh[0][0] == 0 and sh[-1][1] == inter
        assert all(a[1] == b[0] for a, b in zip(sh, sh[1:]))
        assert all((f1 - f0) % 64 == 0 and f1 > f0 for f0, f1 in sh)
        sizes = [f1 - f0 for f0, f1 in sh]
        assert max(sizes) - min(sizes) <= 64
        rows = tp.gate_up_rows(inter, *sh[0])
        assert len(rows) == 2 * (sh[0][1] - sh[0][0]) and rows[len(rows) // 2] == inter + sh[0][0]
    with pytest.raises(ValueError):
        tp.shard_features(100, 2)
    with pytest.raises(ValueError):
        tp.shard_features(128, 3)
