"""Failure detection on the GPU: a pipeline wait that runs out is reported, and
the context stays usable.

Every mbarrier wait of the kernels is bounded by the handle's wait limit
(tt_set_wait_timeout). With a 1 ns limit the waits give up at once: the kernel
sets TT_DEV_WAIT_TIMEOUT, lets the work it issued itself finish (TMA copies,
MMAs and exchange messages, under a separate long bound) and returns. The next
call with the normal limit must then give the oracle's result. Nothing here
traps, faults or hangs: the failure is a wait limit that nothing can meet.

The host-side watchdog tt_sync polls a stream for a bounded time: a stream
kept busy by a bounded spin (torch.cuda._sleep) is reported as still running
within the poll limit, and a commit whose waits gave up shows the status bit
there without clearing it.
"""
import time

import numpy as np
import pytest

from block_diffusion_decoding_attn_b300 import workload as wl

pytestmark = pytest.mark.gpu

DEFAULT_NS = 1_000_000_000


@pytest.fixture(scope="module")
def tt():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_diffusion_decoding_attn_b300 as tt
    from block_diffusion_decoding_attn_b300 import build
    build.build()
    return tt


def _with_tiny_limit(tt, fn):
    import torch
    h = tt.handle(0)
    assert h.get_error() == 0
    h.set_wait_timeout(1)
    try:
        fn()
        torch.cuda.synchronize()
    finally:
        h.set_wait_timeout(DEFAULT_NS)
    return h.get_error()


def test_commit_timeout_reported_then_exact(tt, oracle_lib):
    import torch
    w = wl.custom("timeout_commit", 4, 256, 4, 1, 64, 16, (16,) * 4, V=131072, k=16)
    ci = wl.commit_inputs(w, seed=0)

    def run():
        c = wl.commit_tensors(ci, "cuda")
        tt.commit(c["logits"], w.B, w.L, c["masked"], w.k, c["tok"])

    # tt_get_error (inside) reports the timeout and puts the handle's counters back to zero
    st = _with_tiny_limit(tt, run)
    assert st & tt.TT_DEV_WAIT_TIMEOUT
    c = wl.commit_tensors(ci, "cuda")
    tok, masked = tt.commit(c["logits"], w.B, w.L, c["masked"], w.k, c["tok"])
    torch.cuda.synchronize()
    assert tt.handle(0).get_error() == 0
    ot, om, _, _ = oracle_lib.commit(ci.logits, w.B, w.L, ci.masked, w.k, ci.tok)
    assert np.array_equal(tok.cpu().numpy(), ot)
    assert np.array_equal(masked.cpu().numpy(), om)


def test_attention_timeout_reported_then_exact(tt, oracle_lib):
    import torch
    w = wl.WORKLOADS["b8_c4096_l32"]  # query tiles cut between CTAs, then merged
    inp = wl.attn_inputs(w, seed=0)
    t = wl.attn_tensors(inp)

    def run():
        tt.block_attn(t["q"], t["k_blk"], t["v_blk"], t["k_ctx"], t["v_ctx"], t["ctx_len"])

    st = _with_tiny_limit(tt, run)
    assert st & tt.TT_DEV_WAIT_TIMEOUT
    out = tt.block_attn(t["q"], t["k_blk"], t["v_blk"], t["k_ctx"], t["v_ctx"], t["ctx_len"])
    torch.cuda.synchronize()
    assert tt.handle(0).get_error() == 0
    rows = np.array([[0, 0, 0], [7, 31, 31], [3, 17, 9], [5, 2, 20]], np.int32)
    ref = oracle_lib.block_attn(inp.q, inp.k_blk, inp.v_blk, inp.k_ctx, inp.v_ctx, inp.ctx_len,
                                rows=rows)
    got = out.float().cpu().numpy().astype(np.float64)[rows[:, 0], rows[:, 1], rows[:, 2]]
    assert np.abs(got - ref).max() <= 1e-2 * np.abs(ref).max()


def test_sync_is_bounded_and_reports_without_clearing(tt, oracle_lib):
    import torch
    h = tt.handle(0)
    assert h.get_error() == 0
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        torch.cuda._sleep(1 << 31)  # a bounded spin of 2^31 clocks, about a second
    t0 = time.monotonic()
    done, _ = h.sync(stream=s, timeout_ms=5)
    assert not done and time.monotonic() - t0 < 0.5
    done, st = h.sync(stream=s, timeout_ms=60000)
    assert done and st == 0
    # a commit whose waits give up on the same stream: tt_sync reports the
    # bit and leaves it; tt_get_error then reads and clears it
    w = wl.custom("sync_commit", 4, 256, 4, 1, 64, 16, (16,) * 4, V=131072, k=16)
    ci = wl.commit_inputs(w, seed=1)
    with torch.cuda.stream(s):
        c = wl.commit_tensors(ci, "cuda")
        h.set_wait_timeout(1)
        try:
            tt.commit(c["logits"], w.B, w.L, c["masked"], w.k, c["tok"], stream=s)
            done, st = h.sync(stream=s, timeout_ms=60000)
        finally:
            h.set_wait_timeout(DEFAULT_NS)
    assert done and st & tt.TT_DEV_WAIT_TIMEOUT
    assert h.get_error() & tt.TT_DEV_WAIT_TIMEOUT
    assert h.get_error() == 0
    # and a normal commit on that stream is exact once the stream has drained
    with torch.cuda.stream(s):
        c = wl.commit_tensors(ci, "cuda")
        tok, masked = tt.commit(c["logits"], w.B, w.L, c["masked"], w.k, c["tok"], stream=s)
    done, st = h.sync(stream=s, timeout_ms=60000)
    assert done and st == 0
    ot, om, _, _ = oracle_lib.commit(ci.logits, w.B, w.L, ci.masked, w.k, ci.tok)
    assert np.array_equal(tok.cpu().numpy(), ot)
    assert np.array_equal(masked.cpu().numpy(), om)
