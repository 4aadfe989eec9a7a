"""Shared builders for the GPU parity tests: one seeded workload filled into a
GPU pool through the CUDA append and into a host pool through the oracle's own
append, from the same bf16 rows. Nothing computed by the CUDA path is ever
given to the oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import quantized_paged_kv_cache_gb300 as nk
from quantized_paged_kv_cache_gb300 import workloads as wl

ABS_TOL = 4e-3
REL_L2_TOL = 1e-3


class Built:
    pass


def build(w: wl.Workload, device="cuda", fill=0, chunk=16384, oracle_pool=True, gen_device="cuda"):
    """History (everything except the step's last append_len tokens) plus the
    step's append, appended on both sides in the same chunks."""
    c = Built()
    c.w = w
    c.bt_cpu = wl.block_table(w)
    c.bt = c.bt_cpu.to(device)
    c.ctx = torch.tensor(w.ctx_lens, dtype=torch.int32, device=device)
    c.pool = nk.KVPool.empty(w.num_pages, w.P, w.Hkv, w.D, device=device, fill=fill)
    c.opool = oracle.new_pool(w.num_pages, w.P, w.Hkv, w.D, fill=fill) if oracle_pool else None
    status = torch.zeros(1, dtype=torch.int32, device=device)
    for b in range(w.B):
        L = w.ctx_lens[b]
        pos = 0
        while pos < L:
            n = min(chunk, L - pos)
            k, v = wl.kv_rows(w, b, pos, n, device=gen_device)
            cu = torch.tensor([0, n], dtype=torch.int32)
            # the CUDA append sees only sequence b (B = 1 view of the table)
            nk.kv_append(c.pool, c.bt[b:b + 1].contiguous(), torch.tensor([pos], dtype=torch.int32, device=device),
                         cu.to(device), k.to(device), v.to(device), status=status)
            if oracle_pool:
                rc = oracle.kv_append(c.opool, w.num_pages, w.P, w.Hkv, w.D, c.bt_cpu[b:b + 1], [pos], cu,
                                      k.cpu(), v.cpu())
                assert rc == 0
            pos += n
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    c.q = wl.queries(w, device=gen_device).to(device)
    c.q_cpu = c.q.cpu()
    return c


def gpu_pool_bytes(c) -> np.ndarray:
    return c.pool.storage.cpu().numpy()


def oracle_attention_full(c) -> np.ndarray:
    w = c.w
    return oracle.paged_attention(c.opool, w.num_pages, w.P, w.Hkv, w.D, c.bt_cpu, w.ctx_lens, c.q_cpu, w.T, w.Hq,
                                  w.sm_scale)


def oracle_rows(c, rows) -> np.ndarray:
    """fp64 outputs of the listed (b, t, i) rows."""
    w = c.w
    out = np.empty((len(rows), w.D))
    for j, (b, t, i) in enumerate(rows):
        out[j], _ = oracle.attention_row(c.opool, w.num_pages, w.P, w.Hkv, w.D, c.bt_cpu, w.ctx_lens, c.q_cpu, w.T,
                                         w.Hq, w.sm_scale, b, t, i)
    return out


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    e = np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** -126)))
    return np.exp2(e - 7)


# Elements that needed the |O| >= 2 allowance of compare(), reported at the
# end of the run (tests/conftest.py): [count, largest |O|, largest error].
WIDE = {"elements": 0, "compared": 0, "max_abs_o": 0.0, "max_err": 0.0, "calls": []}


def compare(gpu_bf16: torch.Tensor, ref64: np.ndarray, what=""):
    """Tolerance of a bf16 attention output against the oracle:
    * every element within 4e-3 of the oracle's unrounded fp64 result. A bf16
      number can be that close only where half a bf16 ulp is below 4e-3,
      i.e. |O| < 2; at |O| >= 2 an element may differ by half an ulp (the
      rounding no bf16 output avoids) plus 4e-3. Those elements are counted
      and reported at the end of the run, with their largest magnitude;
    * relative L2 <= 1e-3 against the fp64 result rounded to bf16 (ties to
      even): bf16 rounding alone gives ~1.6e-3 against the unrounded result,
      so that is not the bar for the L2 norm."""
    ref64 = np.asarray(ref64, dtype=np.float64)
    ref = oracle.bits_to_double(oracle.round_bf16(ref64))
    g = gpu_bf16.to(torch.float64).cpu().numpy().reshape(ref.shape)
    x = ref64.reshape(ref.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    err = np.abs(g - x)
    wide = np.abs(x) >= 2.0
    allow = np.where(wide, 0.5 * bf16_ulp(x) + ABS_TOL, ABS_TOL)
    maxabs = float(err.max()) if err.size else 0.0
    worst = float((err / allow).max()) if err.size else 0.0
    rel = float(np.linalg.norm(g - ref) / max(np.linalg.norm(ref), 1e-300))
    rel_exact = float(np.linalg.norm(g - x) / max(np.linalg.norm(x), 1e-300))
    nwide = int(wide.sum())
    WIDE["compared"] += int(err.size)
    if nwide:
        WIDE["elements"] += nwide
        WIDE["max_abs_o"] = max(WIDE["max_abs_o"], float(np.abs(x[wide]).max()))
        WIDE["max_err"] = max(WIDE["max_err"], float(err[wide].max()))
        WIDE["calls"].append(what)
    assert worst <= 1.0, (f"{what}: max-abs {maxabs:.3e} vs the unrounded oracle exceeds 4e-3 "
                          f"(|O| >= 2: half an ulp + 4e-3) (ratio {worst:.2f})")
    assert rel <= REL_L2_TOL, f"{what}: rel-L2 {rel:.3e} > {REL_L2_TOL} (vs unrounded fp64: {rel_exact:.3e})"
    return maxabs, rel, rel_exact


def run_decode(c, impl="mma", num_ctas=0, out=None, status=None, ctx=None, max_ctx=None):
    w = c.w
    fn = nk.paged_decode_attn if impl == "mma" else nk.paged_decode_attn_simt
    return fn(c.pool, c.q, c.bt, c.ctx if ctx is None else ctx, w.sm_scale, w.max_ctx if max_ctx is None else max_ctx,
              num_ctas=num_ctas, out=out, status=status)
