"""Shared helpers of the GPU parity tests: run the library on a case, run the
oracle on the same inputs, compare with the tolerances of the workload
statement (fp32: max-abs 1e-5; bf16 K/V with fp32 accumulation: max-abs 1e-2
beyond the bf16 output's own half-ulp rounding, and relative L2 5e-3). LSE is
compared at 1e-4 absolute (a float32 log-sum-exp of O(1)..O(10) scores), with
-inf matching exactly."""

from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads

TOL = {"f32": {"max_abs": 1e-5}, "bf16": {"max_abs": 1e-2, "rel_l2": 5e-3}}
LSE_ATOL = 1e-4


def as_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy()


def bf16_half_ulp(x: np.ndarray) -> np.ndarray:
    """Half a bf16 unit in the last place at |x|: the rounding error that any
    bf16 result carries against an exact value (8 significant bits)."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.exp2(np.maximum(e, -126.0) - 8.0), 0.0)


def compare(out_gpu, o_ref, dtype, lse_gpu=None, lse_ref=None, what="", margin=1.0):
    """Assert the tolerances; return the max-abs error against them.

    bf16 outputs: the max-abs bound applies to the error beyond the output's
    own rounding, |o - o_ref| - half_ulp_bf16(o_ref) (a bf16 value can be no
    closer to an exact reference than that, e.g. 0.0078 at |o| = 2.5).
    ``margin`` < 1 asks for that fraction of the max-abs bound.
    """
    o = as_f64(out_gpu) if isinstance(out_gpu, torch.Tensor) else out_gpu
    assert np.all(np.isfinite(o)), f"{what}: non-finite output"
    err = np.abs(o - o_ref)
    tol = TOL[dtype]
    if dtype == "bf16":
        err = np.maximum(err - bf16_half_ulp(o_ref), 0.0)
    bound = margin * tol["max_abs"]
    assert err.max() <= bound, f"{what}: max abs err {err.max():.3e} > {bound:.3e}"
    if "rel_l2" in tol:
        rel = np.linalg.norm(o - o_ref) / max(np.linalg.norm(o_ref), 1e-30)
        assert rel <= tol["rel_l2"], f"{what}: rel L2 {rel:.3e} > {tol['rel_l2']}"
    if lse_gpu is not None:
        lg = as_f64(lse_gpu) if isinstance(lse_gpu, torch.Tensor) else lse_gpu
        inf_ref = np.isneginf(lse_ref)
        assert np.array_equal(np.isneginf(lg), inf_ref), f"{what}: -inf LSE mismatch"
        d = np.abs(lg[~inf_ref] - lse_ref[~inf_ref])
        if d.size:
            assert d.max() <= LSE_ATOL, f"{what}: LSE err {d.max():.3e}"
    return float(err.max())


def device_metadata(case: workloads.PagedCase, device="cuda"):
    bt = torch.from_numpy(case.block_table).to(device)
    lens = torch.from_numpy(case.attn_lens).to(device)
    pos = torch.from_numpy(case.positions).to(device)
    return bt, lens, pos


def oracle_decode(case: workloads.PagedCase, seq_idx=None, k_pool=None, v_pool=None):
    """Oracle O/LSE for sequences ``seq_idx`` (pre-append pools + new rows if appending)."""
    v = workloads.oracle_view(case, seq_idx, k_pool=k_pool, v_pool=v_pool)
    kp, vp = v["k_pool"], v["v_pool"]
    if case.append:
        kp, vp = oracle.kv_append(kp, vp, v["k_new"], v["v_new"], v["block_table"], v["positions"],
                                  case.page_size)
    return oracle.decode_attention(v["q"], kp, vp, v["block_table"], v["seq_lens"], case.scale)


def oracle_mla(case: workloads.PagedCase, seq_idx=None):
    """Oracle O/LSE of an absorbed-MLA case for sequences ``seq_idx``."""
    v = workloads.oracle_view(case, seq_idx)
    return oracle.mla_decode_attention(v["q"], v["k_pool"], v["block_table"], v["seq_lens"], case.scale,
                                       case.Dv)
