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
