"""Process-group helpers for the benchmark: one process per GPU, each serving
an independent batch (data-parallel attention: "Step-3 is Large yet
Affordable", section 8.1, each attention GPU processes its own batch), so the
data path has no collective; only the timing is reduced across ranks."""
from __future__ import annotations

import os

import torch
import torch.distributed as dist


def env_rank() -> tuple[int, int, int]:
    """(rank, world_size, local_rank) from the torchrun environment (0, 1, 0 if absent)."""
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def init(backend: str | None = None) -> tuple[int, int, int]:
    rank, world, local = env_rank()
    if world > 1 and not dist.is_initialized():
        if backend is None:
            backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
            dist.init_process_group(backend, device_id=torch.device("cuda", local))
        else:
            dist.init_process_group(backend)
    return rank, world, local


def _device():
    if dist.is_initialized() and dist.get_backend() == "nccl":
        return torch.device("cuda", torch.cuda.current_device())
    return torch.device("cpu")


def barrier():
    if dist.is_initialized():
        if dist.get_backend() == "nccl":
            dist.barrier(device_ids=[torch.cuda.current_device()])
        else:
            dist.barrier()


def reduce_scalar(x: float, op: str) -> float:
    """max or sum of a float over all ranks (identity on one process)."""
    if not dist.is_initialized():
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=_device())
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


def aggregate(bytes_done: float, seconds: float) -> tuple[float, float]:
    """Whole-job throughput: bytes of all ranks over the slowest rank's time.
    Returns (total_bytes, max_seconds)."""
    return reduce_scalar(bytes_done, "sum"), reduce_scalar(seconds, "max")


def aggregate_many(bytes_done, seconds) -> tuple[list, list]:
    """aggregate() for several timed regions at once (one collective per list):
    per region, bytes summed over ranks and the slowest rank's seconds."""
    b = [float(x) for x in bytes_done]
    t = [float(x) for x in seconds]
    if not dist.is_initialized():
        return b, t
    tb = torch.tensor(b, dtype=torch.float64, device=_device())
    tt = torch.tensor(t, dtype=torch.float64, device=_device())
    dist.all_reduce(tb, op=dist.ReduceOp.SUM)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return tb.cpu().tolist(), tt.cpu().tolist()


def finalize():
    if dist.is_initialized():
        dist.destroy_process_group()
