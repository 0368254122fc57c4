"""The allocation-free decode entry point on the GPU (collected last: a failure here stops a -x run only
after every other test has run).

fi_decode_noalloc serves callers that cannot allocate device memory (for
example a runtime that has handed the whole GPU to its own memory pool, or a
plugin whose host forbids allocations): it keeps its plan, page indices, split
counters and partial slots in the library's fixed file-scope device array
instead of a workspace.  These tests call it through the C ABI on different
batches in a row -- so each call finds the previous call's leftovers in the
shared array -- and check every result against the float64 oracle, against
fi_plan + fi_run on a regular workspace, and that the array's error word stays
clear.
"""
import ctypes

import numpy as np
import pytest

from oracle import attention as A
from serving_attention_plan_gb300 import workloads as W

from .gpu_helpers import alloc_out, assert_close, run_library, to_device, torch_mod

pytestmark = pytest.mark.gpu


def _batch(seed, long_len):
    """Decode batch with one long request, so some rows are split across CTAs and merged in-kernel."""
    rng = np.random.default_rng(seed)
    kv = rng.integers(0, 900, size=40)
    kv[3] = long_len
    return W.make_paged_batch(rng, f"noalloc_{seed}", np.ones(40, np.int64), kv, 32, 8, 16, False, pool_pages=None)


def _noalloc(b, dev):
    from serving_attention_plan_gb300 import binding as B
    torch = torch_mod()
    q, k, v = dev
    o, lse = alloc_out(b)
    B.decode_noalloc(b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, b.num_qo_heads, b.num_kv_heads,
                     b.page_size, b.causal, q, k, v, o, lse)
    torch.cuda.synchronize()
    return o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def test_noalloc_matches_oracle_and_workspace_path_on_calls_in_a_row():
    from serving_attention_plan_gb300 import binding as B
    from serving_attention_plan_gb300 import build
    build.build()
    B.decode_noalloc_get_error()  # start from a clear error word
    batches = [_batch(1, 60000), _batch(2, 9000), _batch(1, 60000)]
    for b in batches:
        dev = to_device(b)
        ref_o, ref_lse = A.batch_attention(b)
        ws_o, ws_lse, ws = run_library(b, dev=dev)
        assert ws.info()[7] > 0  # the long request is split, so the scratch slots and counters are used
        o, lse = _noalloc(b, dev)
        assert B.decode_noalloc_get_error() == 0
        assert_close(o, lse, ref_o, ref_lse)
        # the workspace path plans the same way but runs the warp-MMA consumer on these 16-token pages,
        # so the two agree within the parity tolerance (not bit for bit)
        assert_close(o, lse, ws_o, ws_lse)


def test_noalloc_rejects_tensor_core_batches_and_oversize():
    from serving_attention_plan_gb300 import binding as B
    b = W.random_small_batch(5, batch=2, num_qo_heads=8, num_kv_heads=2, page_size=16, causal=True,
                             q_len_range=(20, 30), kv_len_range=(40, 60))
    dev = to_device(b)
    o, lse = alloc_out(b)
    with pytest.raises(B.FiError) as ei:
        B.decode_noalloc(b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, 8, 2, 16, True, *dev, o, lse)
    assert ei.value.status == 3
    # more page ids than the 4 MiB array can hold
    n = 1_200_000
    qo = np.array([0, 1], np.int32)
    kv = np.array([0, n], np.int32)
    idx = np.zeros(n, np.int32)
    with pytest.raises(B.FiError) as ei:
        B.decode_noalloc(qo, kv, idx, np.array([1], np.int32), 8, 2, 1, False, *dev, o, lse)
    assert ei.value.status == 2
    # a KV length above 2^30 (one page id repeated, 2^20-key pages) is rejected by the planner, as by
    # fi_plan; the planner runs before any device work, so the tiny buffers are never read
    ps = 1 << 20
    qo = np.array([0, 1], np.int32)
    kv = np.array([0, 1025], np.int32)
    idx = np.zeros(1025, np.int32)
    last = np.array([ps], np.int32)
    p32 = lambda a: a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
    q, k, v = dev
    st = B.lib().fi_decode_noalloc(p32(qo), p32(kv), p32(idx), p32(last), 1, 8, 2, 128, ps, 0, q.data_ptr(),
                                   k.data_ptr(), v.data_ptr(), 1, o.data_ptr(), lse.data_ptr(), None)
    assert st == 3
    assert B.decode_noalloc_get_error() == 0
