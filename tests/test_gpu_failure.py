"""GPU: failure detection by bounded waits, tested without a GPU fault.

Every wait inside the kernels (mbarrier phases of the TMA rings, the TMEM
accumulators, the side data, the grid barrier of the correction factors) is
bounded: it gives up after its limit, or as soon as another role of the CTA
raised the abort flag, and the kernel then writes S3R_ERR_TIMEOUT to the
caller's status word and exits cleanly.  s3r_debug_wait_timeout runs each
kernel family's own wait routine on an mbarrier that nothing ever arrives on,
with a short limit, so the wait runs out for real; no trap, assert or bad
address is involved, and the context stays usable afterwards.
"""
import pytest
import torch

from parity_util import codes

pytestmark = pytest.mark.gpu

ERR_TIMEOUT = -5   # S3R_ERR_TIMEOUT


@pytest.fixture(scope="module")
def s3r():
    import stochastic_rounding_int8_gb300 as m
    m.lib()
    return m


@pytest.mark.parametrize("family", ["WAIT_GEMM", "WAIT_QUANTIZE", "WAIT_EC"])
def test_wait_runs_out_and_reports(s3r, family):
    """A wait on a phase that never completes gives up after its limit (20 ms
    here, 2 s in the kernels) and reports S3R_ERR_TIMEOUT."""
    limit = 20_000_000
    st, waited = s3r.debug_wait_timeout(getattr(s3r, family), limit)
    assert st == ERR_TIMEOUT
    assert limit <= waited < 20 * limit, waited


@pytest.mark.parametrize("family", ["WAIT_GEMM", "WAIT_EC"])
def test_wait_gives_up_on_the_abort_flag(s3r, family):
    """With a 2 s limit, a wait gives up as soon as another warp of the CTA
    raises the abort flag (about 1 ms in), as the kernels' roles do when one of
    them has given up."""
    st, waited = s3r.debug_wait_timeout(getattr(s3r, family), 2_000_000_000, raise_abort=True)
    assert st == ERR_TIMEOUT
    assert 1_000_000 <= waited < 100_000_000, waited


def test_context_usable_after_timeouts(s3r, orc):
    """After the waits ran out the same context still computes: the S3R
    quantization of a small gradient is bit-exact against the oracle."""
    for fam in (s3r.WAIT_GEMM, s3r.WAIT_QUANTIZE, s3r.WAIT_EC):
        assert s3r.debug_wait_timeout(fam, 5_000_000)[0] == ERR_TIMEOUT
    g = torch.randn(256, 384, generator=torch.Generator().manual_seed(4)) * 1e-3
    gb = g.to(torch.bfloat16)
    st = s3r.new_status()
    q = s3r.s3r_quantize(gb.cuda(), seed=2, tensor_id=5, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    Qo, do, _, _ = orc.quantize(orc.from_torch_bf16(gb), seed=2, tensor_id=5)
    assert (codes(q.Q) == Qo).all()
    assert (q.tile_scale.cpu().numpy() == do).all()


def test_hook_rejects_bad_arguments(s3r):
    L = s3r.lib()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    w = torch.zeros(1, dtype=torch.int64, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert L.s3r_debug_wait_timeout(7, 1000, 0, st.data_ptr(), w.data_ptr(), s) == -1
    assert L.s3r_debug_wait_timeout(0, 0, 0, st.data_ptr(), w.data_ptr(), s) == -1
    assert L.s3r_debug_wait_timeout(0, 3_000_000_000, 0, st.data_ptr(), w.data_ptr(), s) == -1
    assert L.s3r_debug_wait_timeout(1, 1000, 1, st.data_ptr(), w.data_ptr(), s) == -1   # no abort flag there
    assert L.s3r_debug_wait_timeout(0, 1000, 0, None, w.data_ptr(), s) == -1
