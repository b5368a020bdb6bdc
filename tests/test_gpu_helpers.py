"""GPU checks of the measurement and self-check helpers: the FP4 tensor-core
throughput kernel finishes without a device error; a bounded device wait that
nothing completes returns with the TIMEOUT bit and leaves the context usable;
the prefill records its phase events in order (start, append done, then
scored / selected / attended per block)."""
import math

import pytest
import torch

from fp4_compressed_sparse_gb300 import csa2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from fp4_compressed_sparse_gb300 import build_lib
    build_lib.build()
    csa2.load()


def test_mxf4_peak_kernel_runs():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    sink = torch.zeros(sms, dtype=torch.int32, device="cuda")
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    csa2.mxf4_peak_launch(sms, 4096, sink, err)
    b.record()
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    tflops = sms * 4096 * 2.0 * 128 * 128 * 64 / (a.elapsed_time(b) / 1e3) / 1e12
    assert 100.0 < tflops < 40000.0


def test_bounded_wait_timeout_reports_and_returns():
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    csa2.bounded_wait_check(4, True, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0  # completed barrier: the wait succeeds
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    csa2.bounded_wait_check(8, False, err)  # nothing arrives: gives up after 8 polls
    b.record()
    torch.cuda.synchronize()
    assert int(err.item()) == csa2.DEVERR_TIMEOUT
    assert a.elapsed_time(b) < 2000.0
    # the context is intact and the timed-out warp gave its tensor memory back:
    # a tensor-core kernel on every SM allocates all 512 columns and finishes
    err.zero_()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    csa2.mxf4_peak_launch(sms, 64, None, err)
    csa2.bounded_wait_check(1, True, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    x = torch.arange(1024, device="cuda", dtype=torch.float32)
    assert float(x.sum().item()) == 1023 * 1024 / 2


def test_prefill_phase_events(orc):
    from gpu_util import build_r2, cmp_rows
    prior, Q, H_I, H, k = 200, 40, 4, 16, 32
    c, _, rope, err, (ba, bb), _, _ = build_r2(orc, 1, prior, csa2.SWA_MXFP8, seed=3, cap=(prior + Q) // 2 + 8)
    rows = cmp_rows(3, 0, prior, Q)
    g = torch.Generator().manual_seed(4)
    q_idx = torch.randn((Q, H_I, 128), generator=g).to(torch.bfloat16).cuda()
    w = torch.rand((Q, H_I), generator=g).cuda()
    q = torch.randn((Q, H, 576), generator=g).to(torch.bfloat16).cuda()
    idx = torch.empty((Q, k), dtype=torch.int32, device="cuda")
    out = torch.empty((Q, H, 512), device="cuda")
    lse = torch.empty((Q, H), device="cuda")
    ws = csa2.prefill_workspace(Q, c.capacity, H_I, H, k)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(16)]
    for e in ev:
        e.record()
    torch.cuda.synchronize()
    csa2.set_phase_events(ev)
    csa2.prefill_chunk(c, 0, [r.cuda() for r in rows] + [ba.cuda(), bb.cuda()], rope, q_idx, w, q, k,
                       1 / math.sqrt(576), idx, out, lse, ws, err=err)
    n = csa2.phase_events_recorded()
    csa2.set_phase_events(None)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert n == 2 + 3  # one block of 40 queries
    times = [ev[i].elapsed_time(ev[i + 1]) for i in range(n - 1)]
    assert all(t >= 0.0 for t in times)
