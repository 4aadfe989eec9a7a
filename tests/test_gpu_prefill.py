"""GPU parity of the chunked-prefill attention (nk_paged_prefill_attn) against
the fp64 oracle: the T tokens of a prefill chunk attend to the paged INT8 cache
before them and causally to each other ("NInfer-4090" README, "What this fork
changes": the INT8 attention prefill; chunked prefill of 1,024 tokens).

The oracle is the same paged attention definition at large T. Shapes cover
pure prefill (ctx = T), a chunk after history, ragged tails of the 128-row CTA
tiles (G * T not a multiple of 128), head dims 64 / 128 / 256 and page sizes
16 / 32 / 64, garbage past the context, contexts long enough that the output
accumulator is folded into its running total several times, and a full-size
chunk of 1,024 tokens on 8 sequences at 131,072 tokens of context (sampled
rows).
"""
import numpy as np
import pytest
import torch

import oracle
import quantized_paged_kv_cache_gb300 as nk
from quantized_paged_kv_cache_gb300 import workloads as wl

from _cases import build, compare, oracle_attention_full

pytestmark = pytest.mark.gpu

SHAPES = [
    # name, B, T, Hq, Hkv, D, P, ctx_lens
    ("pure_d256", 1, 200, 24, 4, 256, 64, [200]),          # ctx = T: the first chunk
    ("hist_d256", 2, 64, 24, 4, 256, 64, [700, 4099]),      # after history, 12 tiles of 128 rows
    ("tail_d256", 2, 37, 24, 4, 256, 64, [37, 1000]),       # G T = 222: a ragged last tile
    ("d128_p32", 2, 33, 16, 2, 128, 32, [40, 700]),
    ("d64_p16", 1, 100, 2, 1, 64, 16, [300]),
    ("g1_d256", 2, 150, 4, 4, 256, 16, [150, 999]),         # one head per kv-head
    ("t1_d256", 3, 1, 24, 4, 256, 64, [1, 64, 2000]),       # T = 1 through the prefill kernel
    # contexts past the 2,048-key accumulator runs: folds into tensor memory
    ("fold_d128_p16", 1, 48, 16, 2, 128, 16, [6000]),
    ("fold_d64_p32", 2, 20, 4, 1, 64, 32, [2100, 5000]),
]


@pytest.mark.parametrize("shape", SHAPES, ids=[s[0] for s in SHAPES])
@pytest.mark.parametrize("fill", [0, 0xFF])
def test_prefill_matches_oracle(shape, fill):
    name, B, T, Hq, Hkv, D, P, lens = shape
    w = wl.custom(name, B=B, T=T, Hq=Hq, Hkv=Hkv, D=D, P=P, ctx_lens=lens, seed=61,
                  num_pages=sum((L + P - 1) // P for L in lens) + 2, outlier_channels=2, outlier_scale=8.0)
    c = build(w, fill=fill)
    ref = oracle_attention_full(c)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = nk.paged_prefill_attn(c.pool, c.q, c.bt, c.ctx, w.sm_scale, w.max_ctx, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    compare(out, ref, f"{name} fill={fill:#x}")
    again = nk.paged_prefill_attn(c.pool, c.q, c.bt, c.ctx, w.sm_scale, w.max_ctx)
    torch.cuda.synchronize()
    assert torch.equal(out, again), "run-to-run results differ"


@pytest.mark.parametrize("which,s", [("q", -12), ("v", -12), ("v", 10), ("k", 6)])
def test_prefill_scaled_inputs(which, s):
    """Inputs off unit scale: the fp16 operands carry powers of two.

    K moves no fp16 operand (its scales are fp32 and its codes are the same),
    only the size of the scores: at K x 2^10 they reach ~5,000 log2 units,
    where the fp32 sums of the tensor cores (~16 per score) err by a few 1e-3
    in the exponent, enough to move a near-tie by the 4e-3 bar on the 2,304
    rows checked here. K x 2^6 keeps the scores at a few hundred."""
    w = wl.custom(f"pf_{which}{s}", B=1, T=96, Hq=24, Hkv=4, D=256, P=64, ctx_lens=[900], seed=62,
                  **{f"{which}_scale": 2.0 ** s})
    c = build(w)
    ref = oracle_attention_full(c)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = nk.paged_prefill_attn(c.pool, c.q, c.bt, c.ctx, w.sm_scale, w.max_ctx, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    back = 2.0 ** -s if which == "v" else 1.0
    compare(out.to(torch.float64) * back, ref * back, w.name)


def test_prefill_bad_context_is_flagged_and_skipped():
    w = wl.custom("pf_bad", B=2, T=16, Hq=8, Hkv=2, D=128, P=16, ctx_lens=[64, 300], seed=63)
    c = build(w)
    ref = oracle_attention_full(c)
    ctx = c.ctx.clone()
    ctx[0] = 5  # < T
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = nk.paged_prefill_attn(c.pool, c.q, c.bt, ctx, w.sm_scale, w.max_ctx, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & nk.NK_DEVFLAG_BAD_CTX
    compare(out[1], ref[1], "valid sequence next to a bad one")


@pytest.mark.slow
def test_prefill_full_size_chunk():
    """8 sequences, the last 1,024 tokens of 131,072 as the chunk (the
    append + attend mix's shape), in the launch bench.py times; whole pool
    bit-exact after the append, sampled rows against the oracle."""
    from test_gpu_full import build_like_bench
    w = wl.make("mix_prefill")
    pool, opool, bt, bt_cpu = build_like_bench(w)
    assert np.array_equal(pool.storage.cpu().numpy(), opool)
    q = wl.queries(w, device="cuda")
    ctx = torch.tensor(w.ctx_lens, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = nk.paged_prefill_attn(pool, q, bt, ctx, w.sm_scale, w.max_ctx, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rows = [(b, t, i) for b in (0, 7) for t in (0, 511, 1023) for i in (0, 13, 23)]
    q_cpu = q.cpu()
    ref = np.stack([oracle.attention_row(opool, w.num_pages, w.P, w.Hkv, w.D, bt_cpu, w.ctx_lens, q_cpu, w.T, w.Hq,
                                         w.sm_scale, b, t, i)[0] for (b, t, i) in rows])
    got = torch.stack([out[b, t, i] for (b, t, i) in rows])
    compare(got, ref, "mix_prefill")
