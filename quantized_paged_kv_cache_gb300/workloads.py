"""Seeded synthetic workloads (shapes, tables and bf16 inputs), shared by the
tests, the benchmark and the CPU oracle's callers.

This module holds no quantization or attention arithmetic: it only draws
random inputs with the shapes and value structure of the workloads the NInfer
README pages describe (Qwen-27B-class GQA with 24 q-heads over 4 kv-heads and
head_dim 256 -- "NInfer-4090" README, "What this fork changes", the
d256-h24-kv4 shape; 4K..262,144-token depths; concurrency C1..C8; MTP3 verify
with T = 4 columns).

Every random draw comes from a torch.Generator seeded from (config seed,
purpose), so each piece is reproducible on its own. Values are N(0, 1) in fp32
rounded to bf16 (round to nearest even), then shaped per config:
  * c1_decode: 4 fixed K channels per kv-head scaled x8 (outliers that stress
    the group scales);
  * long_context: K and V rows each scaled by an independent U(0.5, 2) factor
    per (token, kv-head) (per-token norm spread);
  * any workload: Q, K or V multiplied by a power of two (q_scale, k_scale,
    v_scale), to move the inputs off unit scale.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass
class Workload:
    name: str
    B: int
    T: int
    Hq: int
    Hkv: int
    D: int
    P: int
    ctx_lens: list[int]
    seed: int
    # tokens each sequence appends in one step (the step's kv_cache_append)
    append_len: int
    # per-config input structure
    outlier_channels: int = 0
    outlier_scale: float = 1.0
    token_norm_range: tuple[float, float] | None = None
    note: str = ""
    # KV format of the pool: "int8" (INT8 group-64, fp32 scales), "rk8v4",
    # "i8f16" (the pages' INT8 layout, fp16 scales) or "bf16" (unquantized)
    fmt: str = "int8"
    # powers of two the drawn Q, K and V values are multiplied by (before the
    # bf16 rounding): the range tests move the inputs off unit scale
    q_scale: float = 1.0
    k_scale: float = 1.0
    v_scale: float = 1.0
    # filled by tables()
    num_pages: int = 0
    max_pages: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def max_ctx(self) -> int:
        return max(self.ctx_lens)

    def pages_of(self, b: int) -> int:
        return (self.ctx_lens[b] + self.P - 1) // self.P

    # stored bytes of one key of one kv-head: int8 K/V codes + fp32 scales per
    # 64 channels (int8); int8 K codes + fp16 scale per 64 channels and 4-bit
    # V codes + fp16 scale per 32 channels (rk8v4)
    def bytes_per_key_head(self) -> int:
        if self.fmt == "rk8v4":
            return self.D + (self.D // 64) * 2 + self.D // 2 + (self.D // 32) * 2
        if self.fmt == "i8f16":
            return 2 * self.D + 2 * (self.D // 64) * 2
        if self.fmt == "bf16":
            return 2 * self.D * 2
        return 2 * self.D + 2 * (self.D // 64) * 4

    # algorithmic bytes of one attention call: the stored K/V of every visible
    # key, bf16 Q read and bf16 O written
    def kv_bytes(self) -> int:
        return sum(self.ctx_lens) * self.Hkv * self.bytes_per_key_head()

    def attn_flops(self) -> int:
        """Multiply-adds x 2 of QK and PV over every visible (query, key) pair."""
        pairs = sum(self.T * (L - self.T) + self.T * (self.T + 1) // 2 for L in self.ctx_lens) * self.Hq
        return 4 * self.D * pairs

    def q_bytes(self) -> int:
        return self.B * self.T * self.Hq * self.D * 2

    def attn_bytes(self) -> int:
        return self.kv_bytes() + 2 * self.q_bytes()

    # algorithmic bytes of one append call: bf16 K and V read, codes and
    # scales written
    def append_rows(self) -> int:
        return self.B * self.append_len

    def append_bytes(self) -> int:
        n = self.append_rows() * self.Hkv
        return n * (2 * self.D * 2 + self.bytes_per_key_head())


def _gen(seed: int, tag: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1_000_003 + tag)
    return g


def make(name: str) -> Workload:
    """The workloads: tiny, c1_decode, c8_verify, long_context, mix,
    c8_decode (the C8 verify contexts at T = 1: plain decode of 8 sequences),
    and c1_rk8v4 (c1_decode's inputs in the rk8v4 format)."""
    if name == "tiny":
        w = Workload("tiny", B=1, T=1, Hq=2, Hkv=1, D=64, P=16, ctx_lens=[256], seed=0, append_len=1,
                     note="1 seq, 1 kv-head, 2 q-heads, head_dim 64, ctx 256, page 16, T=1")
    elif name in ("c1_decode", "c1_rk8v4", "c1_i8f16"):
        fmt = {"c1_rk8v4": "rk8v4", "c1_i8f16": "i8f16"}.get(name, "int8")
        w = Workload(name, B=1, T=1, Hq=24, Hkv=4, D=256, P=64, ctx_lens=[32768], seed=1, append_len=1,
                     outlier_channels=4, outlier_scale=8.0,
                     note="C1 decode: 24 q / 4 kv heads, head_dim 256, ctx 32,768, page 64, T=1, "
                          "4 K outlier channels per head x8", fmt=fmt)
        if fmt != "int8":
            w.note += f"; {fmt} KV format"
    elif name == "c8_i8f16":
        g = _gen(2, 0, "cpu")
        lens = torch.randint(4096, 65536 + 1, (8,), generator=g).tolist()
        w = Workload(name, B=8, T=4, Hq=24, Hkv=4, D=256, P=64, ctx_lens=lens, seed=2, append_len=4,
                     note=f"MTP3 verify C8 (c8_verify's inputs) in the {name[3:]} KV format", fmt=name[3:])
    elif name in ("c8_verify", "c8_decode"):
        g = _gen(2, 0, "cpu")
        lens = torch.randint(4096, 65536 + 1, (8,), generator=g).tolist()
        if name == "c8_verify":
            w = Workload("c8_verify", B=8, T=4, Hq=24, Hkv=4, D=256, P=64, ctx_lens=lens, seed=2, append_len=4,
                         note="MTP3 verify C8: 8 seqs, T=4 causal, ctx ~ U[4,096, 65,536]")
        else:
            w = Workload("c8_decode", B=8, T=1, Hq=24, Hkv=4, D=256, P=64, ctx_lens=lens, seed=2, append_len=1,
                         note="plain decode C8: 8 seqs, T=1, the C8 verify contexts")
    elif name == "long_context":
        w = Workload("long_context", B=1, T=4, Hq=24, Hkv=4, D=256, P=64, ctx_lens=[262144], seed=3, append_len=4,
                     token_norm_range=(0.5, 2.0),
                     note="long context C1: ctx 262,144, T=4 causal, per-token norm x U(0.5, 2)")
    elif name == "mix_prefill":
        w = Workload("mix_prefill", B=8, T=1024, Hq=24, Hkv=4, D=256, P=64, ctx_lens=[131072] * 8, seed=4,
                     append_len=1024,
                     note="the append + attend mix's chunk: 1,024 tokens of each of 8 seqs appended at "
                          "130,048..131,071, then their chunked-prefill attention over 131,072 keys")
    elif name == "prefill_32k":
        w = Workload("prefill_32k", B=2, T=1024, Hq=24, Hkv=4, D=256, P=64, ctx_lens=[32768] * 2, seed=5,
                     append_len=1024,
                     note="a smaller chunked prefill for profiling: 1,024 tokens of each of 2 seqs at "
                          "31,744..32,767, attending to 32,768 keys (142 MB of cache, above the L2)")
    elif name == "mix":
        w = Workload("mix", B=8, T=4, Hq=24, Hkv=4, D=256, P=64, ctx_lens=[131072] * 8, seed=4, append_len=1024,
                     note="append of a 1,024-token chunk into each of 8 seqs (positions 130,048..131,071), "
                          "then C8 x T4 attention at ctx 131,072")
    else:
        raise KeyError(name)
    return tables(w)


CONFIGS = ("tiny", "c1_decode", "c8_verify", "long_context", "mix", "c8_decode")  # INT8 group-64 pools
RK8V4_CONFIGS = ("c1_rk8v4",)
FORMAT_CONFIGS = ("c1_i8f16", "c8_i8f16")  # the pages' INT8 layout (fp16 scales)
PREFILL_CONFIGS = ("mix_prefill", "prefill_32k")  # chunked prefill (T = 1,024)


def tables(w: Workload, num_pages: int | None = None) -> Workload:
    """Block tables: every sequence's pages drawn from one random permutation of the pool."""
    need = sum(w.pages_of(b) for b in range(w.B))
    w.num_pages = num_pages if num_pages is not None else need
    w.max_pages = max(w.pages_of(b) for b in range(w.B))
    perm = torch.randperm(w.num_pages, generator=_gen(w.seed, 1, "cpu")).to(torch.int32)
    bt = torch.full((w.B, w.max_pages), -1, dtype=torch.int32)
    off = 0
    for b in range(w.B):
        n = w.pages_of(b)
        bt[b, :n] = perm[off:off + n]
        off += n
    w.extra["block_table"] = bt
    return w


def custom(name="custom", *, B, T, Hq, Hkv, D, P, ctx_lens, seed, append_len=None, num_pages=None,
           outlier_channels=0, outlier_scale=1.0, token_norm_range=None, q_scale=1.0, k_scale=1.0,
           v_scale=1.0) -> Workload:
    w = Workload(name, B=B, T=T, Hq=Hq, Hkv=Hkv, D=D, P=P, ctx_lens=list(ctx_lens), seed=seed,
                 append_len=T if append_len is None else append_len, outlier_channels=outlier_channels,
                 outlier_scale=outlier_scale, token_norm_range=token_norm_range, q_scale=q_scale, k_scale=k_scale,
                 v_scale=v_scale)
    return tables(w, num_pages)


def block_table(w: Workload) -> torch.Tensor:
    return w.extra["block_table"]


def outlier_index(w: Workload) -> torch.Tensor:
    """[Hkv][outlier_channels] K channel indices scaled by outlier_scale."""
    if w.outlier_channels == 0:
        return torch.zeros((w.Hkv, 0), dtype=torch.long)
    g = _gen(w.seed, 2, "cpu")
    return torch.stack([torch.randperm(w.D, generator=g)[: w.outlier_channels] for _ in range(w.Hkv)])


def kv_rows(w: Workload, b: int, start: int, n: int, device="cpu") -> tuple[torch.Tensor, torch.Tensor]:
    """bf16 K and V rows [n][Hkv][D] for positions start .. start+n-1 of sequence b.

    Rows are drawn per (sequence, 4096-position block) so any sub-range is
    reproducible independently of how the caller slices it."""
    blk = 4096
    ks, vs = [], []
    first, last = start // blk, (start + n - 1) // blk if n > 0 else start // blk - 1
    oi = outlier_index(w)
    for k in range(first, last + 1):
        g = _gen(w.seed, 1000 + b * 100_000 + k, device)
        kk = torch.randn((blk, w.Hkv, w.D), generator=g, device=device, dtype=torch.float32)
        vv = torch.randn((blk, w.Hkv, w.D), generator=g, device=device, dtype=torch.float32)
        if w.outlier_channels:
            for h in range(w.Hkv):
                kk[:, h, oi[h].to(device)] *= w.outlier_scale
        if w.token_norm_range is not None:
            lo, hi = w.token_norm_range
            uk = torch.rand((blk, w.Hkv, 1), generator=g, device=device) * (hi - lo) + lo
            uv = torch.rand((blk, w.Hkv, 1), generator=g, device=device) * (hi - lo) + lo
            kk *= uk
            vv *= uv
        a = max(start, k * blk) - k * blk
        e = min(start + n, (k + 1) * blk) - k * blk
        ks.append((kk[a:e] * w.k_scale).to(torch.bfloat16))
        vs.append((vv[a:e] * w.v_scale).to(torch.bfloat16))
    if not ks:
        z = torch.empty((0, w.Hkv, w.D), dtype=torch.bfloat16, device=device)
        return z, z.clone()
    return torch.cat(ks).contiguous(), torch.cat(vs).contiguous()


def queries(w: Workload, device="cpu") -> torch.Tensor:
    """bf16 Q [B][T][Hq][D]."""
    g = _gen(w.seed, 3, device)
    q = torch.randn((w.B, w.T, w.Hq, w.D), generator=g, device=device, dtype=torch.float32)
    return (q * w.q_scale).to(torch.bfloat16)


def history_and_step(w: Workload):
    """(prior lengths, step start positions): the step appends the last
    append_len tokens of every sequence; everything before is history."""
    starts = [L - w.append_len for L in w.ctx_lens]
    return starts, starts


def append_batch(w: Workload, starts: list[int], lens: list[int], device="cpu"):
    """Concatenated rows for an append call: (k, v, start_pos int32 [B], cu_new int32 [B+1])."""
    ks, vs, cu = [], [], [0]
    for b in range(w.B):
        k, v = kv_rows(w, b, starts[b], lens[b], device)
        ks.append(k)
        vs.append(v)
        cu.append(cu[-1] + lens[b])
    k = torch.cat(ks).contiguous() if ks else torch.empty((0, w.Hkv, w.D), dtype=torch.bfloat16)
    v = torch.cat(vs).contiguous() if vs else torch.empty((0, w.Hkv, w.D), dtype=torch.bfloat16)
    return k, v, torch.tensor(starts, dtype=torch.int32), torch.tensor(cu, dtype=torch.int32)
