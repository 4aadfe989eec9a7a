"""The allocation-free decode entry point (GPU).

nk_paged_decode_attn_noalloc serves callers that cannot allocate device
memory (a host that owns a fixed device budget and forbids cudaMalloc after
start, or code that must not risk the synchronization an allocation can
bring): it keeps the split partials in a fixed array owned by the library
instead of a caller-provided workspace. Called twice in a row through the C
ABI, it must give bit for bit the output of the regular entry point at the
same split count (both run the same kernels), stay within the attention
tolerance of the fp64 oracle, and leave the device's free memory unchanged.
This file sorts last so a failure here comes after every other test has run;
it also passes on its own in a fresh process (the first call on a device sets
up the array's address).
"""
import pytest
import torch

import quantized_paged_kv_cache_gb300 as nk
from quantized_paged_kv_cache_gb300 import workloads as wl

from _cases import build, compare, oracle_attention_full

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape", [
    ("noalloc_t4", 3, 4, 24, 4, 256, 64, [700, 4099, 33]),
    ("noalloc_t1", 2, 1, 8, 2, 128, 16, [1000, 17]),
])
def test_noalloc_matches_workspace_entry(shape):
    name, B, T, Hq, Hkv, D, P, lens = shape
    w = wl.custom(name, B=B, T=T, Hq=Hq, Hkv=Hkv, D=D, P=P, ctx_lens=lens, seed=77,
                  num_pages=sum((L + P - 1) // P for L in lens) + 2)
    c = build(w)
    # B = 0 performs only the per-device set-up (the warm-up before a capture)
    nk.paged_decode_attn_noalloc(c.pool, c.q[:0], c.bt, c.ctx, w.sm_scale, w.max_ctx)
    ref = nk.paged_decode_attn(c.pool, c.q, c.bt, c.ctx, w.sm_scale, w.max_ctx)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = [torch.full_like(c.q, float("nan")) for _ in range(2)]
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    alloc0 = torch.cuda.memory_allocated()
    for call in range(2):
        nk.paged_decode_attn_noalloc(c.pool, c.q, c.bt, c.ctx, w.sm_scale, w.max_ctx, out=outs[call], status=status)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_allocated() == alloc0
    assert free1 == free0, f"device free memory changed by {free0 - free1} bytes"
    assert int(status.item()) == 0
    ref64 = oracle_attention_full(c)
    for call in range(2):
        assert torch.equal(outs[call].view(torch.int16), ref.view(torch.int16)), f"{name} call {call}"
        compare(outs[call], ref64, f"{name} call {call} vs oracle")


def test_noalloc_rejects_shapes_beyond_its_array():
    w = wl.custom("noalloc_big", B=1, T=4, Hq=24, Hkv=4, D=256, P=16, ctx_lens=[64], seed=3)
    c = build(w, oracle_pool=False)
    # 5000 CTAs need (5000 + 4) * 24 * 257 * 4 bytes of partials: more than the array holds
    need = nk.decode_workspace_bytes(1, 4, 24, 4, 256, 5000)
    assert need > nk.NOALLOC_MAX_WORKSPACE
    with pytest.raises(nk.NKError) as ei:
        nk.paged_decode_attn_noalloc(c.pool, c.q, c.bt, c.ctx, w.sm_scale, w.max_ctx, num_ctas=5000)
    assert ei.value.code == 4
