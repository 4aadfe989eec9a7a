"""The tcgen05 decode's folding instance against the fp64 oracle (GPU).

When one CTA may run more than 512 pages of one kv-head through its fp32
PV accumulators, the host takes the instance of the split kernel that folds
them into a tensor-memory total every 128 pages (the accumulation error of
mma.sync grows with the products one accumulator takes in). One CTA over a
ragged 547-page sequence followed by a short one runs four folds, a
partial last run and a segment change with the total reset. Shapes cover
the three tile shapes of the kernel (12, 24 and 30 rows per kv-head) and
both scale layouts (fp32 scales; the pages' fp16 scales, "NInfer-3090"
README, "Choosing a KV format"). The default split of the same inputs runs
the unfolded instance and must agree with the oracle too.
"""
import pytest
import torch

import quantized_paged_kv_cache_gb300 as nk
from quantized_paged_kv_cache_gb300 import workloads as wl

from _cases import build, compare, oracle_attention_full
from test_gpu_formats import build_fmt, oracle_out

pytestmark = pytest.mark.gpu

LENS = [547 * 64 - 37, 1000]


@pytest.mark.parametrize("T", [2, 4, 5])
def test_fold_instance_int8(T):
    w = wl.custom(f"fold_t{T}", B=2, T=T, Hq=6, Hkv=1, D=256, P=64, ctx_lens=LENS, seed=31,
                  num_pages=sum((L + 63) // 64 for L in LENS) + 2)
    c = build(w)
    ref = oracle_attention_full(c)
    for n in (1, 0):  # one CTA: folding instance; default split: unfolded
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        out = nk.paged_decode_attn(c.pool, c.q, c.bt, c.ctx, w.sm_scale, w.max_ctx, num_ctas=n, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        compare(out, ref, f"{w.name}/ctas={n}")


@pytest.mark.parametrize("T", [4, 5])
def test_fold_instance_i8f16(T):
    w = wl.custom(f"fold_i8f16_t{T}", B=2, T=T, Hq=6, Hkv=1, D=256, P=64, ctx_lens=LENS, seed=32,
                  num_pages=sum((L + 63) // 64 for L in LENS) + 2)
    c = build_fmt("i8f16", w)
    assert c.status == 0
    ref = oracle_out("i8f16", c)
    for n in (1, 0):
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        out = nk.i8f16_decode_attn(c.pool, c.q, c.bt, c.ctx, w.sm_scale, w.max_ctx, num_ctas=n, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        compare(out, ref, f"{w.name}/ctas={n}")


def test_fold_instance_in_column_chunks():
    # T = 12 at G = 6: three launches of 4 columns, each over the same pages
    # with its own causal limits, each taking the folding instance in one CTA
    w = wl.custom("fold_t12", B=2, T=12, Hq=6, Hkv=1, D=256, P=64, ctx_lens=LENS, seed=33,
                  num_pages=sum((L + 63) // 64 for L in LENS) + 2)
    c = build(w)
    ref = oracle_attention_full(c)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = nk.paged_decode_attn(c.pool, c.q, c.bt, c.ctx, w.sm_scale, w.max_ctx, num_ctas=1, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    compare(out, ref, f"{w.name}/ctas=1")


def test_fold_instance_in_the_step_call():
    # nk_decode_step: the step's rows (the last T of each sequence, appended
    # again with the same values) and the attention, one CTA
    T = 4
    w = wl.custom("fold_step", B=2, T=T, Hq=6, Hkv=1, D=256, P=64, ctx_lens=LENS, seed=34,
                  num_pages=sum((L + 63) // 64 for L in LENS) + 2)
    c = build(w)
    ref = oracle_attention_full(c)
    rows = [wl.kv_rows(w, b, L - T, T, device="cuda") for b, L in enumerate(LENS)]
    k = torch.cat([r[0] for r in rows]).contiguous()
    v = torch.cat([r[1] for r in rows]).contiguous()
    start = torch.tensor([L - T for L in LENS], dtype=torch.int32, device="cuda")
    cu = torch.tensor([0, T, 2 * T], dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = nk.decode_step(c.pool, c.bt, start, cu, k, v, c.q, c.ctx, w.sm_scale, w.max_ctx, num_ctas=1, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    compare(out, ref, f"{w.name}/ctas=1")
