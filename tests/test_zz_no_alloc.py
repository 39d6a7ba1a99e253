"""tt_commit_noalloc against tt_commit, through the C ABI, on the GPU.

tt_commit_noalloc is for callers that cannot allocate device memory (a
serving engine that has reserved all of HBM for its own pool, a plug-in host
that forbids allocation while a request runs): its scratch is a fixed array
inside the library instead of a handle's allocated scratch. It must give
exactly what tt_commit gives (committed ids and mask, bit for bit) call after
call, even though every call reuses the same scratch.

This file is collected last on purpose, and passes both alone in a fresh
process and after the other tests.
"""
import ctypes

import pytest

from block_diffusion_decoding_attn_b300 import workload as wl

pytestmark = pytest.mark.gpu

_P = ctypes.c_void_p


@pytest.fixture(scope="module")
def tt():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_diffusion_decoding_attn_b300 import build
    build.build()
    import block_diffusion_decoding_attn_b300 as tt
    return tt


def _status(tt) -> int:
    st = ctypes.c_int(-1)
    rc = tt.lib().tt_commit_noalloc_status(ctypes.byref(st))
    assert rc == 0, tt.lib().tt_last_error()
    return st.value


def test_noalloc_matches_commit_on_two_calls_in_a_row(tt):
    import torch
    w = wl.WORKLOADS["b8_c4096_l32"]
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    m_ref = torch.ones(w.rows, dtype=torch.uint8, device=dev)   # tt_commit path
    t_ref = torch.full((w.rows,), -1, dtype=torch.int32, device=dev)
    m_na, t_na = m_ref.clone(), t_ref.clone()                     # allocation-free path
    for call in range(2):  # the second call starts from the first call's outputs
        lg = torch.from_numpy(wl.logits(w, seed=3, step=call)).to(dev)
        mo_ref = torch.empty_like(m_ref)
        tt.commit(lg, w.B, w.L, m_ref, w.k, t_ref, masked_out=mo_ref)
        mo_na = torch.empty_like(m_na)
        rc = tt.lib().tt_commit_noalloc(_P(lg.data_ptr()), w.B, w.L, w.V, _P(m_na.data_ptr()),
                                        w.k, _P(t_na.data_ptr()), _P(mo_na.data_ptr()),
                                        _P(stream.cuda_stream))
        assert rc == 0, tt.lib().tt_last_error()
        torch.cuda.synchronize()
        assert torch.equal(t_na, t_ref), f"token ids differ after call {call}"
        assert torch.equal(mo_na, mo_ref), f"mask differs after call {call}"
        m_ref, m_na = mo_ref, mo_na
    assert int((m_na == 0).sum()) == 2 * w.k * w.B
    assert _status(tt) == 0  # no wait timed out


def test_noalloc_at_its_row_limit_in_place(tt):
    # B*L = 65536, the scratch's bound: the highest key/prediction/ticket
    # offsets and the block selection for L > 256, the mask updated in place,
    # two calls in a row
    import torch
    w = wl.custom("limit", 256, 256, 1, 1, 8, 8, (0,) * 256, V=1024, k=16)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    m0 = torch.from_numpy(wl.random_mask(w, 0.7, seed=8)).to(dev)
    m_ref, m_na = m0.clone(), m0.clone()
    t_ref = torch.full((w.rows,), -1, dtype=torch.int32, device=dev)
    t_na = t_ref.clone()
    for call in range(2):
        lg = torch.from_numpy(wl.logits(w, seed=9, step=call)).to(dev)
        tt.commit(lg, w.B, w.L, m_ref, w.k, t_ref, masked_out=m_ref)
        rc = tt.lib().tt_commit_noalloc(_P(lg.data_ptr()), w.B, w.L, w.V, _P(m_na.data_ptr()),
                                        w.k, _P(t_na.data_ptr()), _P(m_na.data_ptr()),
                                        _P(stream.cuda_stream))
        assert rc == 0, tt.lib().tt_last_error()
        torch.cuda.synchronize()
        assert torch.equal(t_na, t_ref), f"token ids differ after call {call}"
        assert torch.equal(m_na, m_ref), f"mask differs after call {call}"
    assert _status(tt) == 0


def test_noalloc_rejects_sizes_beyond_its_scratch(tt):
    import torch
    x = torch.zeros(16, dtype=torch.float32, device="cuda")
    rc = tt.lib().tt_commit_noalloc(_P(x.data_ptr()), 257, 256, 4, _P(x.data_ptr()), 1,
                                    _P(x.data_ptr()), _P(x.data_ptr()), None)
    assert rc == -2
    assert b"65536" in tt.lib().tt_last_error()
