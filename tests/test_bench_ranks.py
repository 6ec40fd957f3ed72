"""The multi-rank host logic of bench.py on CPU: two gloo ranks (independent
replicas) agree on the slowest rank's time and on the whole-job throughput."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out_dir):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = bench.max_over_ranks(100.0 + 25.0 * rank, world, device="cpu")
    tok = bench.job_tokens_per_s(2400, world, ms)
    dist.barrier()
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"r{rank}"), "w") as f:
        f.write(f"{ms} {tok}")


@pytest.mark.parametrize("world", [2])
def test_max_over_ranks_and_job_throughput(tmp_path, world):
    mp.spawn(_rank, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    got = [tuple(map(float, open(tmp_path / f"r{r}").read().split())) for r in range(world)]
    slowest = 100.0 + 25.0 * (world - 1)
    for ms, tok in got:
        assert ms == slowest
        assert tok == pytest.approx(world * 2400 / (slowest / 1000.0))


def test_single_rank_needs_no_collective():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5


def test_launch_counts_of_the_decode_paths():
    """bench.py's gpu_launches claim per step, on a stand-in stack: the
    35b stack's two-kernel chain is the layer-0 router and its top-K, A and
    B per layer and one ranking launch (83); its cluster form is the router,
    the top-K, one launch per layer, the output sum and the ranking (44); the
    single self-predicting tiny layer needs no router."""
    import sys
    from types import SimpleNamespace
    sys.path.insert(0, ROOT)
    import bench
    from int4_expert_gemv_gb300.configs import ALL, TINY

    def stand_in(shared_gu_rank):
        lora = [SimpleNamespace(r=0) for _ in range(3)]
        shared = [SimpleNamespace(r=shared_gu_rank) for _ in range(3)]
        ed = SimpleNamespace(lora=lora, shared_lora=shared)
        return SimpleNamespace(chain=True, fused=True, m=SimpleNamespace(layers=[{"experts_desc": ed}]))

    assert bench.kernels_per_step(ALL["35b"], stand_in(16)) == 83
    assert bench.kernels_per_step(ALL["35b"], stand_in(16), cluster=True) == 44
    assert bench.kernels_per_step(TINY, stand_in(0)) == 3
    assert bench.kernels_per_step(TINY, stand_in(0), cluster=True) == 3
