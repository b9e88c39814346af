"""A whole step captured once in a CUDA graph and replayed gives the eager
step's result bit for bit: the library's calls launch kernels only (no
allocation, host synchronisation or pageable copy once the workspace is
sized), so a serving loop can capture its per-step calls.  Decode (append
fused into the split pass, then the merge) and chunked prefill (append, then
the prefill kernel)."""
import pytest
import torch

from paged_kv_cache_253_gb300 import runtime, workloads as wls

from gpu_common import run_library

pytestmark = pytest.mark.gpu

D128 = dict(num_q_heads=32, num_kv_heads=8, head_dim=128)


def _capture_and_replay(step):
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):                     # warm-up off the default stream
        step.run()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = step.out.clone()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step.run()
    step.out.zero_()
    graph.replay()
    graph.replay()                                    # replays leave the work counters reset
    torch.cuda.synchronize()
    return eager


def test_decode_step_replays_from_a_graph():
    wl = wls.make_workload("decode", num_seqs=8, min_len=1, max_len=700, **D128)
    values = wls.generate_values(wl, "cuda")
    pool, _, _, step = run_library(wl, values)
    assert pool.get_error() == 0
    first = step.out.clone()
    eager = _capture_and_replay(step)
    assert pool.get_error() == 0
    assert torch.equal(eager, first)                  # re-appending the same token is idempotent
    assert torch.equal(step.out, eager)


def test_prefill_step_replays_from_a_graph():
    wl = wls.make_workload("prefill", lengths=[0, 37, 300], chunks=[90, 5, 140], **D128)
    values = wls.generate_values(wl, "cuda")
    pool, bm, _ = runtime.replay_setup(wl, values, "cuda")
    step = runtime.prepare_prefill(wl, values, pool, bm)
    step.run()
    torch.cuda.synchronize()
    assert pool.get_error() == 0
    first = step.out.clone()
    eager = _capture_and_replay(step)
    assert pool.get_error() == 0
    assert torch.equal(eager, first) and torch.equal(step.out, eager)
