"""Full-size parity on the benchmark workloads, in the launch
configuration bench.py times (default CTA count, the step's append as one
batched call).

Codes and scales are compared bit-exactly over the whole pool; the attention
output is compared on sampled rows the oracle computes one by one (first and
last verify column, first, last and a middle q-head, of every sequence)."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import quantized_paged_kv_cache_gb300 as nk
from quantized_paged_kv_cache_gb300 import workloads as wl

from _cases import compare

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def build_like_bench(w):
    """History appended per sequence in 16K-token chunks, then the step's
    append of every sequence in one call (as bench.py does), on both sides."""
    dev = "cuda"
    bt_cpu = wl.block_table(w)
    bt = bt_cpu.to(dev)
    pool = nk.KVPool.empty(w.num_pages, w.P, w.Hkv, w.D, device=dev, fill=0)
    opool = oracle.new_pool(w.num_pages, w.P, w.Hkv, w.D)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    hist, _ = wl.history_and_step(w)
    for b in range(w.B):
        pos = 0
        while pos < hist[b]:
            n = min(16384, hist[b] - pos)
            k, v = wl.kv_rows(w, b, pos, n, device=dev)
            cu = torch.tensor([0, n], dtype=torch.int32)
            nk.kv_append(pool, bt[b:b + 1].contiguous(), torch.tensor([pos], dtype=torch.int32, device=dev),
                         cu.to(dev), k, v, status=status)
            assert oracle.kv_append(opool, w.num_pages, w.P, w.Hkv, w.D, bt_cpu[b:b + 1], [pos], cu, k.cpu(),
                                    v.cpu()) == 0
            pos += n
    starts, _ = wl.history_and_step(w)
    k, v, sp, cu = wl.append_batch(w, starts, [w.append_len] * w.B, device=dev)
    nk.kv_append(pool, bt, sp.to(dev), cu.to(dev), k, v, status=status)
    assert oracle.kv_append(opool, w.num_pages, w.P, w.Hkv, w.D, bt_cpu, sp, cu, k.cpu(), v.cpu()) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return pool, opool, bt, bt_cpu


@pytest.mark.parametrize("name", wl.CONFIGS)
@pytest.mark.parametrize("impl", ["mma", "simt"])
def test_full_size(name, impl):
    if impl == "simt" and name in ("long_context", "mix"):
        pytest.skip("CUDA-core kernel is checked on the three smaller workloads")
    w = wl.make(name)
    pool, opool, bt, bt_cpu = build_like_bench(w)
    assert np.array_equal(pool.storage.cpu().numpy(), opool), "codes/scales differ from the oracle"
    q = wl.queries(w, device="cuda")
    ctx = torch.tensor(w.ctx_lens, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    fn = nk.paged_decode_attn if impl == "mma" else nk.paged_decode_attn_simt
    out = fn(pool, q, bt, ctx, w.sm_scale, w.max_ctx, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rows = []
    for b in range(w.B):
        for t in sorted({0, w.T - 1}):
            for i in sorted({0, min(w.Hq // 2 + 1, w.Hq - 1), w.Hq - 1}):
                rows.append((b, t, i))
    q_cpu = q.cpu()
    ref = np.stack([oracle.attention_row(opool, w.num_pages, w.P, w.Hkv, w.D, bt_cpu, w.ctx_lens, q_cpu, w.T, w.Hq,
                                         w.sm_scale, b, t, i)[0] for (b, t, i) in rows])
    got = torch.stack([out[b, t, i] for (b, t, i) in rows])
    maxabs, rel, rel_exact = compare(got, ref, f"{name}/{impl}")
    log = os.environ.get("NK_PARITY_LOG")
    if log:
        with open(log, "a") as f:
            f.write(json.dumps({"workload": name, "kernel": impl, "rows": len(rows), "max_abs": maxabs,
                                "rel_l2_vs_bf16_oracle": rel, "rel_l2_vs_fp64_oracle": rel_exact,
                                "codes_scales": "bit-exact", "pool_bytes": int(pool.storage.numel())}) + "\n")


@pytest.fixture(scope="module")
def long_pool():
    w = wl.make("long_context")
    return (w,) + build_like_bench(w)


# (T, CTAs): 4 CTAs over one 262,144-key sequence put 4,096 pages of one
# kv-head through one CTA's PV accumulators; T = 2 and 4 run the tcgen05
# kernel (its folding instance), T = 1 the mma.sync kernel.
@pytest.mark.parametrize("T,ctas", [(1, 4), (2, 4), (4, 4), (4, 16)])
def test_coarse_split_long_context(long_pool, T, ctas):
    w0, pool, opool, bt, bt_cpu = long_pool
    w = wl.custom(f"long_T{T}", B=1, T=T, Hq=w0.Hq, Hkv=w0.Hkv, D=w0.D, P=w0.P, ctx_lens=w0.ctx_lens, seed=17)
    q = wl.queries(w, device="cuda")
    ctx = torch.tensor(w.ctx_lens, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = nk.paged_decode_attn(pool, q, bt, ctx, w.sm_scale, w.max_ctx, num_ctas=ctas, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rows = [(0, w.T - 1, i) for i in range(w.Hq)]
    q_cpu = q.cpu()
    ref = np.stack([oracle.attention_row(opool, w0.num_pages, w.P, w.Hkv, w.D, bt_cpu, w.ctx_lens, q_cpu, w.T, w.Hq,
                                         w.sm_scale, b, t, i)[0] for (b, t, i) in rows])
    got = torch.stack([out[b, t, i] for (b, t, i) in rows])
    compare(got, ref, f"long_context T={T} ctas={ctas}")
