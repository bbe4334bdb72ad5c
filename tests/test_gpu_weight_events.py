"""Ordering of the weight writes against another stream (dmuon_set_weight_events).

A copy of step k's weights runs on a second stream: it waits for the event the library records after
step k's last launch that writes W, and records the event that step k+1 waits on before its first
launch that writes W. The copy is held back by a bounded spin on its stream, so that step k+1 would
overwrite W under it if it did not wait. Every copy must then hold exactly the weights after step k,
and the steps must give the same bits as synchronous steps without events."""

import pytest
import torch

from matrix_optimizer_update_gb300.inputs import random_matrix

from helpers import LibRun

pytestmark = pytest.mark.gpu

SHAPES = [(1024, 4096), (4096, 1024), (1408, 2048), (512, 512), (300, 700)]


def fill(run, seed):
    for i, (r, c) in enumerate(run.shapes):
        run.set(i, W=random_matrix(r, c, seed + 3 * i, 0.02, "cuda", run.param),
                G=random_matrix(r, c, seed + 3 * i + 1, 1e-3, "cuda", run.grad),
                M=random_matrix(r, c, seed + 3 * i + 2, 1e-3, "cuda", "f32"))


@pytest.mark.parametrize("ns_steps", [5, 0])
def test_weight_copies_wait_for_and_hold_back_the_weight_writes(ns_steps):
    steps = 3
    a = LibRun(SHAPES, ns_steps=ns_steps, capture=False)  # with the events
    b = LibRun(SHAPES, ns_steps=ns_steps, capture=False)  # synchronous reference
    fill(a, 8100)
    b.W.copy_(a.W)
    b.G.copy_(a.G)
    b.M.copy_(a.M)
    ref = []
    for _ in range(steps):
        b.step()
        torch.cuda.synchronize()
        ref.append(b.W.clone())

    main, side = torch.cuda.Stream(), torch.cuda.Stream()
    w_ready, w_copied = torch.cuda.Event(), torch.cuda.Event()
    w_ready.record(main)  # creates both events
    w_copied.record(side)
    plan = a.muon.plan
    plan.set_weight_events(w_copied.cuda_event, w_ready.cuda_event)
    copies = [torch.empty_like(a.W) for _ in range(steps)]
    torch.cuda.synchronize()
    for k in range(steps):
        plan.step(a.ptrs(a.W), a.ptrs(a.G), a.ptrs(a.M), 0.02, 0.95, True, main.cuda_stream)
        with torch.cuda.stream(side):
            side.wait_event(w_ready)
            torch.cuda._sleep(50_000_000)  # a bounded spin (tens of ms) ahead of the copy
            copies[k].copy_(a.W, non_blocking=True)
            w_copied.record(side)
    torch.cuda.synchronize()
    plan.set_weight_events(0, 0)
    assert plan.read_device_status(main.cuda_stream) == 0
    for k in range(steps):
        assert torch.equal(copies[k], ref[k]), k
    assert torch.equal(a.M, b.M)

    # cleared events: the next step runs as before
    a.step()
    b.step()
    torch.cuda.synchronize()
    assert torch.equal(a.W, b.W)
