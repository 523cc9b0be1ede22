"""Repeated launches on one workspace: the kernels whose CTAs wait on one
another (request barriers and polls in the selection, split tickets in the
attention, cluster barriers in the latent-row attention) keep their status
word at 0 and give bit-identical results launch after launch.  A race
between CTAs shows up here as a wait that runs out or a result that
changes, which a single parity launch can miss."""
import math

import numpy as np
import pytest
import torch

import skvtest as T
import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def skv():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from sparse_kv_long_gb300 import _build
    _build.build()
    import sparse_kv_long_gb300 as m
    return m


def _repeat(launch, outputs, status, reps, check_every=50):
    launch()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    first = [o.clone() for o in outputs]
    for r in range(reps):
        launch()
        if r % check_every == check_every - 1:
            torch.cuda.synchronize()
            assert int(status.item()) == 0, f"status {int(status.item())} after {r + 2} launches"
            for o, f in zip(outputs, first):
                assert torch.equal(o, f), f"result changed after {r + 2} launches"


@pytest.fixture(scope="module")
def sketch_workload(skv):
    import bench
    w = bench.SketchWorkloadGPU(torch, skv, wl, torch.device("cuda", 0), layers=1)
    yield w
    torch.cuda.synchronize()


def test_layer_step_repeated(skv, sketch_workload):
    """The chained layer step at 8 x 250,000 (append, fold, score + select,
    known-rows attention), 300 times with the same inputs: the append
    rewrites the same row, so every launch gives the same picks and output."""
    w = sketch_workload
    _repeat(lambda: w.layer_step(0), [w.idx, w.cnt, w.out[0]], w.status, 300)


def test_separate_calls_repeated(skv, sketch_workload):
    """The same layer through the separate calls (prepare, score + select,
    the attention in its plain mode), 300 times."""
    w = sketch_workload
    _repeat(lambda: w.layer(0), [w.idx, w.cnt, w.out[0]], w.status, 300)


def test_mla_repeated(skv):
    """Latent-row attention, 32 requests x 2,048 rows (two splits per
    request merged inside a cluster of four), 200 launches on one workspace."""
    B, n_pool, rows_per = 32, 8192, 2048
    x = wl.mla_inputs_cpu(B, n_pool, seed=5)
    rng = np.random.default_rng(6)
    rows = np.stack([np.sort(rng.choice(n_pool, rows_per, replace=False)) for _ in range(B)]).astype(np.int32)
    count = np.full((B,), rows_per, np.int32)
    q, pool, r, cnt = T.bf16_dev(x["q"]), T.dev(x["pool"]), T.dev(rows), T.dev(count)
    out = torch.zeros((B, 128, 512), dtype=torch.float32, device="cuda")
    ws = torch.zeros((max(16, skv.mla_workspace_size(B, rows_per)),), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")

    def launch():
        skv.sparse_attend_mla(q, pool, r, cnt, 1 / math.sqrt(576), out, ws, status=st)

    _repeat(launch, [out], st, 200)
