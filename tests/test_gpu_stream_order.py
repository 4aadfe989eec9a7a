"""Stream order of dependent calls.

Every kernel of the library is launched with programmatic stream
serialization, so it may become resident while the previous kernel of the
stream still runs; each kernel waits for its predecessor (griddepcontrol.wait)
before its first global-memory access. These tests enqueue chains of dependent
calls with no host synchronization in between -- append then decode, step
after step, on one shared workspace (the next split kernel overwrites the
partials the previous combine reads) -- eagerly and as a captured CUDA graph,
and compare every step's output with the oracle run step by step. The same
chains run through nk_decode_step, whose split kernel reads its lengths,
block-table entries and Q while the step's append still runs.
"""
import numpy as np
import pytest
import torch

import oracle
import quantized_paged_kv_cache_gb300 as nk
from quantized_paged_kv_cache_gb300 import workloads as wl

from _cases import build, compare

pytestmark = pytest.mark.gpu

STEPS = 6


def chain_case(T, lens, seed):
    # the pool and the block table cover the contexts after all steps
    P = 64
    final = [L + STEPS * T for L in lens]
    w = wl.custom("chain", B=len(lens), T=T, Hq=24, Hkv=4, D=256, P=P, ctx_lens=final, seed=seed,
                  num_pages=sum((L + P - 1) // P for L in final) + 3)
    hist = wl.custom("chain", B=len(lens), T=T, Hq=24, Hkv=4, D=256, P=P, ctx_lens=lens, seed=seed,
                     num_pages=w.num_pages)
    hist.extra["block_table"] = w.extra["block_table"][:, :hist.max_pages].contiguous()
    c = build(hist, fill=0)
    c.w_final = w
    c.bt_full_cpu = wl.block_table(w)
    c.bt_full = c.bt_full_cpu.cuda()
    return c


def step_inputs(c, i):
    """Rows appended and queries of step i (positions L_i .. L_i + T - 1)."""
    w = c.w_final
    T = w.T
    starts = [L + i * T for L in c.w.ctx_lens]
    k, v, sp, cu = wl.append_batch(w, starts, [T] * w.B)
    g = torch.Generator().manual_seed(7000 + i)
    q = torch.randn((w.B, T, w.Hq, w.D), generator=g).to(torch.bfloat16)
    ctx = [s + T for s in starts]
    return k, v, sp, cu, q, ctx


def oracle_steps(c):
    w = c.w_final
    opool = c.opool.copy()
    refs = []
    for i in range(STEPS):
        k, v, sp, cu, q, ctx = step_inputs(c, i)
        assert oracle.kv_append(opool, w.num_pages, w.P, w.Hkv, w.D, c.bt_full_cpu, sp, cu, k, v) == 0
        refs.append(oracle.paged_attention(opool, w.num_pages, w.P, w.Hkv, w.D, c.bt_full_cpu, ctx, q, w.T, w.Hq,
                                           w.sm_scale))
    return refs


def device_inputs(c):
    ins = []
    for i in range(STEPS):
        k, v, sp, cu, q, ctx = step_inputs(c, i)
        ins.append(dict(k=k.cuda(), v=v.cuda(), sp=sp.cuda(), cu=cu.cuda(), q=q.cuda(),
                        ctx=torch.tensor(ctx, dtype=torch.int32, device="cuda"), max_ctx=max(ctx)))
    return ins


def enqueue(c, ins, ws, outs, status, stream, fused=False, num_ctas=0):
    """Append + attention per step: two calls, or one nk_decode_step (fused)."""
    w = c.w_final
    for i, a in enumerate(ins):
        if fused:
            nk.decode_step(c.pool, c.bt_full, a["sp"], a["cu"], a["k"], a["v"], a["q"], a["ctx"], w.sm_scale,
                           a["max_ctx"], num_ctas=num_ctas, workspace=ws, out=outs[i], status=status, stream=stream)
            continue
        nk.kv_append(c.pool, c.bt_full, a["sp"], a["cu"], a["k"], a["v"], status=status, stream=stream)
        nk.paged_decode_attn(c.pool, a["q"], c.bt_full, a["ctx"], w.sm_scale, a["max_ctx"], num_ctas=num_ctas,
                             workspace=ws, out=outs[i], status=status, stream=stream)


def workspace(c):
    w = c.w_final
    return torch.empty(nk.decode_workspace_bytes(w.B, w.T, w.Hq, w.Hkv, w.D), dtype=torch.uint8, device="cuda")


# T = 1 runs the mma.sync kernel, T = 2 (12 rows per kv-head) the tcgen05
# kernel, T = 8 (48 rows) two tcgen05 column chunks
@pytest.mark.parametrize("fused", [False, True], ids=["two_calls", "decode_step"])
@pytest.mark.parametrize("T,lens", [(1, [130, 2000]), (2, [63, 1500, 700]), (8, [8, 600])], ids=["t1", "t2", "t8"])
def test_chained_steps_match_oracle(T, lens, fused):
    c = chain_case(T, lens, seed=40 + T)
    refs = oracle_steps(c)
    ins = device_inputs(c)
    ws = workspace(c)
    outs = [torch.empty_like(a["q"]) for a in ins]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    enqueue(c, ins, ws, outs, status, torch.cuda.current_stream(), fused=fused)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for i in range(STEPS):
        compare(outs[i], refs[i], f"step {i}")


@pytest.mark.parametrize("T,lens", [(1, [130, 2000]), (2, [63, 1500, 700]), (4, [5, 640]), (8, [9, 400])],
                         ids=["t1", "t2", "t4", "t8"])
def test_decode_step_equals_two_calls(T, lens):
    """nk_decode_step leaves the same pool bytes and the same outputs, bit for
    bit, as nk_kv_append followed by nk_paged_decode_attn (same CTA count)."""
    c = chain_case(T, lens, seed=90 + T)
    w = c.w_final
    n = nk.decode_default_ctas(w.B, w.Hkv, max(a for a in w.ctx_lens), w.P)
    ins = device_inputs(c)
    ws = workspace(c)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    hist = c.pool.storage.clone()
    res = {}
    for fused in (False, True):
        c.pool.storage.copy_(hist)
        outs = [torch.empty_like(a["q"]) for a in ins]
        enqueue(c, ins, ws, outs, status, torch.cuda.current_stream(), fused=fused, num_ctas=n)
        torch.cuda.synchronize()
        res[fused] = (c.pool.storage.clone(), outs)
    assert int(status.item()) == 0
    assert torch.equal(res[False][0], res[True][0]), "pool bytes differ"
    for i in range(STEPS):
        assert torch.equal(res[False][1][i], res[True][1][i]), f"step {i} output differs"


@pytest.mark.parametrize("fused", [False, True], ids=["two_calls", "decode_step"])
def test_graph_replay_matches_eager(fused):
    """The same chain captured once into a CUDA graph: a replay on a pool reset
    to the history gives bit-identical outputs and pool bytes to the eager run."""
    c = chain_case(1, [100, 900], seed=77)
    ins = device_inputs(c)
    ws = workspace(c)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    hist = c.pool.storage.clone()
    eager = [torch.empty_like(a["q"]) for a in ins]
    enqueue(c, ins, ws, eager, status, torch.cuda.current_stream(), fused=fused)
    torch.cuda.synchronize()
    pool_eager = c.pool.storage.clone()

    c.pool.storage.copy_(hist)
    outs = [torch.zeros_like(a["q"]) for a in ins]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            enqueue(c, ins, ws, outs, status, s, fused=fused)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    for rep in range(2):
        c.pool.storage.copy_(hist)
        for o in outs:
            o.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(c.pool.storage, pool_eager), f"replay {rep}: pool bytes differ"
        for i in range(STEPS):
            assert torch.equal(outs[i], eager[i]), f"replay {rep}: step {i} output differs"
    refs = oracle_steps(c)
    for i in range(STEPS):
        compare(outs[i], refs[i], f"graph step {i}")


@pytest.mark.parametrize("T,lens", [(1, [130, 2000]), (4, [5, 640])], ids=["t1", "t4"])
def test_host_step_equals_device_step(T, lens):
    """nk_decode_step_host (inputs from one pinned host buffer, output and
    status read back, the stream waited for) leaves the same pool bytes and
    returns the same outputs, bit for bit, as nk_decode_step on device copies
    of the same inputs, step after step; and the outputs match the oracle."""
    c = chain_case(T, lens, seed=120 + T)
    w = c.w_final
    refs = oracle_steps(c)
    n = nk.decode_default_ctas(w.B, w.Hkv, max(a for a in w.ctx_lens), w.P)
    ins = device_inputs(c)
    ws = workspace(c)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    hist = c.pool.storage.clone()
    # device path
    outs = [torch.empty_like(a["q"]) for a in ins]
    enqueue(c, ins, ws, outs, status, torch.cuda.current_stream(), fused=True, num_ctas=n)
    torch.cuda.synchronize()
    pool_dev = c.pool.storage.clone()
    # host path
    c.pool.storage.copy_(hist)
    total = int(ins[0]["k"].shape[0])
    nbytes, offs = nk.step_host_layout(w.B, total, T, w.Hq, w.Hkv, w.D)
    staging = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    out_dev = torch.empty_like(ins[0]["q"])
    st_h = torch.zeros(1, dtype=torch.int32).pin_memory()
    for i, a in enumerate(ins):
        h_in = torch.zeros(nbytes, dtype=torch.uint8).pin_memory()
        for name, o in zip(("k", "v", "q", "sp", "cu", "ctx"), offs):
            t = a[name]
            nb = t.numel() * t.element_size()
            h_in[o:o + nb].view(t.dtype).view(t.shape).copy_(t.cpu())
        out_h = torch.empty(a["q"].shape, dtype=a["q"].dtype).pin_memory()
        nk.decode_step_host(c.pool, c.bt_full, w.B, total, T, w.Hq, w.sm_scale, a["max_ctx"], h_in, staging, out_dev,
                            out_h, num_ctas=n, workspace=ws, status=status, status_host=st_h)
        assert int(st_h.item()) == 0
        assert torch.equal(out_h, outs[i].cpu()), f"step {i}: host-step output differs"
        compare(out_h.cuda(), refs[i], f"host step {i}")
    assert torch.equal(c.pool.storage, pool_dev), "pool bytes differ"
