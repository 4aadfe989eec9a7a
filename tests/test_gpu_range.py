"""The tensor-core kernels on inputs far from unit scale (GPU).

The method is scale-free: with K scaled by a power of two the cache holds the
same codes with scaled scales, and Q or K scaled changes the scores, not the
range the kernels may use; with V scaled by 2^s the output is 2^s times the
output at unit scale. fp16 operands are not scale-free (normal range 2^-14 ..
65504), so the tensor-core kernels carry powers of two beside them. These
cases scale Q, K and V one at a time by 2^-12 and 2^10, on a shape of the
tcgen05 kernel (T = 4, 24 query rows per kv-head) and of the mma.sync kernel
(T = 1), and a full-size C8 x T4 verify with V x 2^-12, against the oracle run
on the same scaled inputs. A V-scaled output is compared after both it and the
oracle's are multiplied by 2^-s (exact in either), so the 4e-3 bound keeps its
meaning; the device status must stay 0 (no range flag).
"""
import numpy as np
import pytest
import torch

import oracle
import quantized_paged_kv_cache_gb300 as nk
from quantized_paged_kv_cache_gb300 import workloads as wl

from _cases import build, compare, oracle_attention_full

pytestmark = pytest.mark.gpu

SHAPES = {
    # name: (B, T, Hq, Hkv, D, P, ctx_lens)
    "t4_d256": (2, 4, 24, 4, 256, 64, [700, 4099]),
    "t1_d256": (1, 1, 24, 4, 256, 64, [1000]),
    "t2_d128": (2, 2, 16, 2, 128, 32, [33, 515]),
}


@pytest.mark.parametrize("shape", list(SHAPES))
@pytest.mark.parametrize("which", ["q", "k", "v"])
@pytest.mark.parametrize("s", [-12, 10])
def test_scaled_inputs(shape, which, s):
    B, T, Hq, Hkv, D, P, lens = SHAPES[shape]
    scales = {f"{which}_scale": 2.0 ** s}
    w = wl.custom(f"{shape}_{which}{s}", B=B, T=T, Hq=Hq, Hkv=Hkv, D=D, P=P, ctx_lens=lens, seed=31,
                  num_pages=sum((L + P - 1) // P for L in lens) + 3, **scales)
    c = build(w)
    ref = oracle_attention_full(c)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for fn in (nk.paged_decode_attn, nk.paged_decode_attn_simt):
        out = fn(c.pool, c.q, c.bt, c.ctx, w.sm_scale, w.max_ctx, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, f"device status {int(status.item())}"
        back = 2.0 ** -s if which == "v" else 1.0
        compare((out.to(torch.float64) * back), ref * back, f"{w.name}/{fn.__name__}")


def test_full_size_c8_verify_values_scaled_down():
    """The C8 x T4 verify workload (tcgen05 kernel, default CTA count) with V
    x 2^-12: the whole pool bit-exact, sampled rows within tolerance."""
    w = wl.make("c8_verify")
    w.v_scale = 2.0 ** -12
    from test_gpu_full import build_like_bench
    pool, opool, bt, bt_cpu = build_like_bench(w)
    assert np.array_equal(pool.storage.cpu().numpy(), opool)
    q = wl.queries(w, device="cuda")
    ctx = torch.tensor(w.ctx_lens, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = nk.paged_decode_attn(pool, q, bt, ctx, w.sm_scale, w.max_ctx, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rows = [(b, t, i) for b in range(w.B) for t in (0, w.T - 1) for i in (0, 13, w.Hq - 1)]
    q_cpu = q.cpu()
    ref = np.stack([oracle.attention_row(opool, w.num_pages, w.P, w.Hkv, w.D, bt_cpu, w.ctx_lens, q_cpu, w.T, w.Hq,
                                         w.sm_scale, b, t, i)[0] for (b, t, i) in rows])
    got = torch.stack([out[b, t, i] for (b, t, i) in rows]).to(torch.float64) * 2.0 ** 12
    compare(got, ref * 2.0 ** 12, "c8_verify V x 2^-12")
