"""Failure detection of the decode and prefill kernels' bounded waits (GPU),
without a fault: the copies of some pages are simply never issued.

nk_test_inject_copy_stall makes the tensor-core kernels skip the page
copies of CTA page numbers >= k and bounds every wait by a short limit. A wait
for such a page runs out: the call must report NK_DEVFLAG_TIMEOUT in the
status word, return within a fraction of a second, and leave the device
usable -- the next, normal call on the same pool gives the oracle's result.
Nothing is left in flight: the kernels wait for the copies and tensor-core
work they did issue before they exit.
"""
import time

import pytest
import torch

import quantized_paged_kv_cache_gb300 as nk
from quantized_paged_kv_cache_gb300 import workloads as wl

from _cases import build, compare, oracle_attention_full

pytestmark = pytest.mark.gpu

SHAPES = {
    # the tcgen05 kernel (T = 4, 24 rows per kv-head) and the mma.sync kernel (T = 1)
    "tc_t4": (2, 4, 24, 4, 256, 64, [2100, 900]),
    "mma_t1": (2, 1, 24, 4, 256, 64, [2100, 900]),
    "mma_d128": (2, 2, 16, 2, 128, 32, [1500, 700]),
}
WAIT = 1 << 20  # cycles (~0.5 ms)


@pytest.fixture(autouse=True)
def no_injection_left():
    yield
    nk.test_inject_copy_stall(-1)


@pytest.mark.parametrize("shape", list(SHAPES))
@pytest.mark.parametrize("withheld", [0, 2])
def test_withheld_copies_time_out_and_the_device_recovers(shape, withheld):
    B, T, Hq, Hkv, D, P, lens = SHAPES[shape]
    w = wl.custom(shape, B=B, T=T, Hq=Hq, Hkv=Hkv, D=D, P=P, ctx_lens=lens, seed=55,
                  num_pages=sum((L + P - 1) // P for L in lens) + 1)
    c = build(w)
    ref = oracle_attention_full(c)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    # few CTAs, so that every CTA has more pages than the withheld index
    nk.paged_decode_attn(c.pool, c.q, c.bt, c.ctx, w.sm_scale, w.max_ctx, num_ctas=4, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    nk.test_inject_copy_stall(withheld, WAIT)
    t0 = time.perf_counter()
    nk.paged_decode_attn(c.pool, c.q, c.bt, c.ctx, w.sm_scale, w.max_ctx, num_ctas=4, status=status)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    nk.test_inject_copy_stall(-1)
    assert int(status.item()) & nk.NK_DEVFLAG_TIMEOUT, f"status {int(status.item())}: no timeout reported"
    assert elapsed < 1.0, f"the call took {elapsed:.3f} s"
    # the device and the pool are still usable
    status.zero_()
    out = nk.paged_decode_attn(c.pool, c.q, c.bt, c.ctx, w.sm_scale, w.max_ctx, num_ctas=4, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    compare(out, ref, f"{shape} after the timed-out call")


def test_decode_step_reports_the_timeout():
    """The one-call step: the append runs, the attention's waits run out."""
    B, T, Hq, Hkv, D, P, lens = SHAPES["tc_t4"]
    w = wl.custom("step_timeout", B=B, T=T, Hq=Hq, Hkv=Hkv, D=D, P=P, ctx_lens=lens, seed=56,
                  num_pages=sum((L + P - 1) // P for L in lens) + 1)
    c = build(w)
    starts = [L - T for L in lens]
    k, v, sp, cu = wl.append_batch(w, starts, [T] * B, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    nk.test_inject_copy_stall(1, WAIT)
    nk.decode_step(c.pool, c.bt, sp.cuda(), cu.cuda(), k, v, c.q, c.ctx, w.sm_scale, w.max_ctx, num_ctas=4,
                   status=status)
    torch.cuda.synchronize()
    nk.test_inject_copy_stall(-1)
    st = int(status.item())
    assert st & nk.NK_DEVFLAG_TIMEOUT, f"status {st}: no timeout reported"
    assert st & ~(nk.NK_DEVFLAG_TIMEOUT | nk.NK_DEVFLAG_RANGE) == 0, f"status {st}"


def test_prefill_reports_the_timeout_and_the_device_recovers():
    """The chunked prefill's page ring: copies of the CTAs' pages 2 and on are
    withheld; the call reports the timeout quickly (a non-finite output may be
    flagged too: the stages hold stale bytes), and the next call gives the
    oracle's result."""
    w = wl.custom("pf_timeout", B=1, T=64, Hq=8, Hkv=2, D=128, P=32, ctx_lens=[1500], seed=57,
                  num_pages=(1500 + 31) // 32 + 1)
    c = build(w)
    ref = oracle_attention_full(c)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    nk.paged_prefill_attn(c.pool, c.q, c.bt, c.ctx, w.sm_scale, w.max_ctx, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    nk.test_inject_copy_stall(2, WAIT)
    t0 = time.perf_counter()
    nk.paged_prefill_attn(c.pool, c.q, c.bt, c.ctx, w.sm_scale, w.max_ctx, status=status)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    nk.test_inject_copy_stall(-1)
    st = int(status.item())
    assert st & nk.NK_DEVFLAG_TIMEOUT, f"status {st}: no timeout reported"
    assert st & ~(nk.NK_DEVFLAG_TIMEOUT | nk.NK_DEVFLAG_RANGE) == 0, f"status {st}"
    assert elapsed < 1.0, f"the call took {elapsed:.3f} s"
    status.zero_()
    out = nk.paged_prefill_attn(c.pool, c.q, c.bt, c.ctx, w.sm_scale, w.max_ctx, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    compare(out, ref, "prefill after the timed-out call")
