"""Shared helpers of the GPU parity tests: device upload, library calls, comparison."""
import numpy as np

# Tolerances of the parity bar: bf16 inputs, fp32 accumulation, bf16 output.
O_ATOL = 2e-2
LSE_RTOL = 1e-3


def torch_mod():
    import torch
    return torch


def to_device(b):
    torch = torch_mod()
    dev = torch.device("cuda", 0)
    cvt = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
    return cvt(b.q), cvt(b.k_pages), cvt(b.v_pages)


def alloc_out(b):
    torch = torch_mod()
    o = torch.full((b.total_q, b.num_qo_heads, b.head_dim), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((b.total_q, b.num_qo_heads), float("nan"), dtype=torch.float32, device="cuda")
    return o, lse


def run_library(b, num_sms=0, ws=None, dev=None, out=None):
    """Plan + run through the C ABI; returns (o, lse) as float64 numpy plus the workspace."""
    from serving_attention_plan_gb300 import binding as B
    torch = torch_mod()
    if ws is None:
        ws = B.Workspace(b.batch_size, max(b.total_q, 1), max(int(b.kv_indptr[-1]), 1), b.num_qo_heads,
                         b.num_kv_heads, b.head_dim, num_sms)
    q, k, v = dev if dev is not None else to_device(b)
    o, lse = out if out is not None else alloc_out(b)
    ws.plan(b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, b.page_size, b.causal)
    ws.run(q, k, v, o, lse)
    torch.cuda.synchronize()
    assert ws.get_error() == 0
    return o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64), ws


def assert_close(o, lse, ref_o, ref_lse, rows=None):
    """Element-wise parity: |dO| <= 2e-2 absolute, |dLSE| <= 1e-3 * max(1, |LSE|), -inf exactly."""
    if rows is not None:
        o, lse, ref_o, ref_lse = o[rows], lse[rows], ref_o[rows], ref_lse[rows]
    assert not np.isnan(o).any(), "unwritten or NaN output rows"
    assert not np.isnan(lse).any(), "unwritten or NaN LSE rows"
    empty = np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(lse), empty), "empty rows differ"
    err_o = np.abs(o - ref_o).max(initial=0.0)
    assert err_o <= O_ATOL, f"max |dO| = {err_o}"
    fin = ~empty
    if fin.any():
        rel = np.abs(lse[fin] - ref_lse[fin]) / np.maximum(1.0, np.abs(ref_lse[fin]))
        assert rel.max() <= LSE_RTOL, f"max rel |dLSE| = {rel.max()}"
    assert np.all(o[empty] == 0)
    return err_o
